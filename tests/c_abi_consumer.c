/* A plain C consumer of the library's C ABI (include/moe_ep.h): no Python, no PyTorch.
 * Test fixture for tests/test_gpu_c_abi.py.
 *
 *   c_abi_consumer N T H E R payload(0 bf16, 1 fp8) x.bin idx.bin w.bin out.bin
 *
 * Reads the bf16 tokens [N][T][H], int32 expert ids [N][T][R] and fp32 weights [N][T][R],
 * allocates every device buffer itself (cudaMalloc: the library allocates nothing), runs
 * moe_layout_init, moe_forward (then the same pass through moe_dispatch and moe_combine in
 * token batches, which must match) and moe_status_sync on its own stream, and writes the bf16
 * output [N][T][H]. Exit status 0 on success, else the step that failed on stderr. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "moe_ep.h"

static int read_file(const char *path, void *dst, size_t bytes) {
    FILE *f = fopen(path, "rb");
    if (!f) return 0;
    size_t got = fread(dst, 1, bytes, f);
    fclose(f);
    return got == bytes;
}

static void *dev(size_t bytes) {
    void *p = NULL;
    if (cudaMalloc(&p, bytes ? bytes : 16) != cudaSuccess) return NULL;
    return p;
}

#define CHECK(cond, what)                                   \
    do {                                                    \
        if (!(cond)) {                                      \
            fprintf(stderr, "c_abi_consumer: %s\n", what);  \
            return 1;                                       \
        }                                                   \
    } while (0)

int main(int argc, char **argv) {
    CHECK(argc == 11, "usage: N T H E R payload x.bin idx.bin w.bin out.bin");
    moe_dims d;
    d.N = atoi(argv[1]);
    d.T = atoi(argv[2]);
    d.H = atoi(argv[3]);
    d.E = atoi(argv[4]);
    d.R = atoi(argv[5]);
    d.cap = 0;
    d.payload = atoi(argv[6]) ? MOE_PAYLOAD_FP8_E4M3_B128 : MOE_PAYLOAD_BF16;
    CHECK(moe_check_dims(&d) == MOE_OK, "moe_check_dims");

    const size_t tok = (size_t)d.N * d.T, pairs = tok * d.R, L = (size_t)d.E / d.N;
    const size_t B = moe_row_bytes(&d), RB = moe_recv_capacity_rows(&d), cap = (size_t)moe_capacity(&d);
    const size_t xb = tok * d.H * 2;
    uint16_t *hx = (uint16_t *)malloc(xb), *hout = (uint16_t *)malloc(xb);
    int32_t *hidx = (int32_t *)malloc(pairs * 4);
    float *hw = (float *)malloc(pairs * 4);
    CHECK(hx && hout && hidx && hw, "host allocation");
    CHECK(read_file(argv[7], hx, xb) && read_file(argv[8], hidx, pairs * 4) && read_file(argv[9], hw, pairs * 4),
          "reading the inputs");

    cudaStream_t s;
    CHECK(cudaStreamCreate(&s) == cudaSuccess, "cudaStreamCreate");
    const size_t ws_bytes = moe_layout_workspace_bytes(&d);
    void *ws = dev(ws_bytes);
    moe_buffers_t b;
    b.x = (uint16_t *)dev(xb);
    b.xq = (uint8_t *)dev(tok * B);
    b.idx = (int32_t *)dev(pairs * 4);
    b.w = (float *)dev(pairs * 4);
    b.send = dev(pairs * B);
    b.recv = dev((size_t)d.N * RB * B);
    b.expert_x = dev((size_t)d.N * L * cap * (d.payload == MOE_PAYLOAD_BF16 ? B : (size_t)d.H));
    b.expert_scale = d.payload == MOE_PAYLOAD_BF16 ? NULL : (float *)dev((size_t)d.N * L * cap * (d.H / 128) * 4);
    b.expert_y = (uint16_t *)dev((size_t)d.N * L * cap * d.H * 2);
    b.csend = (uint16_t *)dev((size_t)d.N * RB * d.H * 2);
    b.crecv = (uint16_t *)dev(pairs * d.H * 2);
    b.out = (uint16_t *)dev(xb);
    CHECK(ws && b.x && b.xq && b.idx && b.w && b.send && b.recv && b.expert_x && b.expert_y && b.csend && b.crecv &&
              b.out && (d.payload == MOE_PAYLOAD_BF16 || b.expert_scale),
          "cudaMalloc");

    moe_layout_t lay;
    CHECK(moe_layout_init(&d, ws, ws_bytes, &lay, s) == MOE_OK, "moe_layout_init");
    CHECK(cudaMemcpyAsync(b.x, hx, xb, cudaMemcpyHostToDevice, s) == cudaSuccess, "copy x");
    CHECK(cudaMemcpyAsync(b.idx, hidx, pairs * 4, cudaMemcpyHostToDevice, s) == cudaSuccess, "copy idx");
    CHECK(cudaMemcpyAsync(b.w, hw, pairs * 4, cudaMemcpyHostToDevice, s) == cudaSuccess, "copy w");
    moe_status st = moe_forward(&d, &lay, &b, s);
    CHECK(st == MOE_OK, moe_status_string(st));
    uint32_t bits = 0;
    st = moe_status_sync(&lay, s, &bits);
    CHECK(st == MOE_OK, moe_status_string(st));
    CHECK(cudaMemcpy(hout, b.out, xb, cudaMemcpyDeviceToHost) == cudaSuccess, "copy out");

    /* The same pass through the whole-phase calls, in 3 token batches each: the layout,
     * moe_dispatch, the identity expert, moe_combine; the output must equal moe_forward's. */
    lay.batches = 3;
    CHECK(moe_batches(&d, &lay, 2) == (d.T < 3 ? d.T : 3), "moe_batches");
    uint16_t *out2 = (uint16_t *)dev(xb), *hout2 = (uint16_t *)malloc(xb);
    CHECK(out2 && hout2, "second output");
    st = moe_layout(&d, b.idx, &lay, s);
    if (st == MOE_OK) st = moe_dispatch(&d, &lay, b.x, b.send, b.recv, b.expert_x, b.expert_scale, s);
    if (st == MOE_OK) st = moe_expert_identity(&d, &lay, b.expert_x, b.expert_scale, b.expert_y, s);
    if (st == MOE_OK) st = moe_combine(&d, &lay, b.expert_y, b.csend, b.crecv, b.w, out2, s);
    CHECK(st == MOE_OK, moe_status_string(st));
    st = moe_status_sync(&lay, s, &bits);
    CHECK(st == MOE_OK, moe_status_string(st));
    CHECK(cudaMemcpy(hout2, out2, xb, cudaMemcpyDeviceToHost) == cudaSuccess, "copy out2");
    CHECK(memcmp(hout, hout2, xb) == 0, "moe_dispatch + moe_combine differ from moe_forward");

    FILE *f = fopen(argv[10], "wb");
    CHECK(f && fwrite(hout, 1, xb, f) == xb, "writing the output");
    fclose(f);
    printf("launches %llu\n", (unsigned long long)moe_launch_count());
    return 0;
}
