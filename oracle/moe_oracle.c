/*
 * CPU oracle for MoE expert-parallel dispatch and combine.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark may load this library. The product (the CUDA library) never calls it,
 * and the two share no code: no headers, no helpers, no constants.
 *
 * Plain, slow and direct: every function below is the defining formula written out as
 * nested loops over source rank s, destination rank d, token t, routed slot k and
 * hidden element h. Nothing is blocked, fused or reordered beyond what the definition
 * states. Floating point is fp32 with separate multiply and add (build with
 * -ffp-contract=off) plus an fp64 variant of the combine sum.
 *
 * Source: "Enabling trillion-parameter models on AWS EFA" (Perplexity, 2025-11-04),
 * sections "MoE all-to-all over EFA", "Send and receive buffers", "Dispatch and
 * combine" and "Evaluation". The pages print no formulas; the readings this oracle
 * takes where they are silent are:
 *   - expert e lives on rank owner(e) = e / L with local index e % L, L = E / N;
 *   - a rank's send buffer is ordered by (expert, token, slot), so each destination
 *     rank receives one contiguous slice ("a single write per peer");
 *   - a rank's receive buffer holds the slices of source ranks 0..N-1 in order;
 *   - expert l's grouped rows are ordered by (source rank, token, slot);
 *   - the "weighted average" of combine is the plain sum of w * y over the R experts
 *     (router weights already sum to one), accumulated in fp32 in slot order and
 *     rounded once to bf16;
 *   - block-scaled fp8: 128-element blocks, scale = amax / 448 (1 when amax is 0),
 *     q = e4m3(x / scale) rounded to nearest even with saturation to +-448.
 * Status bits returned: 1<<2 expert id out of [0,E), 1<<3 expert capacity exceeded,
 * 1<<4 receive bound exceeded.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BIT_EXPERT_RANGE (1u << 2)
#define ORC_BIT_CAPACITY (1u << 3)
#define ORC_BIT_RECV_BOUND (1u << 4)

/* ---------------------------------------------------------------- number formats */

/* bf16 -> fp32: the bf16 bits are the top half of the fp32 bits. */
float orc_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even (NaN -> quiet NaN with the same sign). */
uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* Round a non-negative double with few significant bits to the nearest integer, ties
 * to even. */
static double rne_int(double v) {
    double f = floor(v);
    double r = v - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* OCP 8-bit floating point, E4M3: sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * No infinities; S.1111.111 is NaN; the largest finite magnitude is 1.75 * 2^8 = 448;
 * exponent field 0 holds subnormals m * 2^-9. */
double orc_e4m3_decode(uint8_t c) {
    int sign = (c >> 7) & 1;
    int ex = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (ex == 15 && m == 7) return NAN;
    if (ex == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + (double)m / 8.0, ex - 7);
    return sign ? -v : v;
}

/* fp32 -> E4M3, round to nearest even, finite values beyond +-448 saturate to +-448.
 * NaN maps to the positive NaN code 0x7F. */
uint8_t orc_e4m3_encode(float f) {
    if (isnan(f)) return 0x7F;
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal grid, step 2^-9; a result of 8 is 2^-6, whose code is 0x08 */
        double q = rne_int(a * 512.0);
        return (uint8_t)(sign | (uint8_t)q);
    }
    int e2;
    frexp(a, &e2);             /* a in [2^(e2-1), 2^e2) */
    int ue = e2 - 1;           /* unbiased exponent, -6..8 */
    double q = rne_int(ldexp(a, 3 - ue)); /* 8..16: 1.mmm scaled by 8 */
    int ef = ue + 7;
    int m = (int)q - 8;
    if (m == 8) {
        ef += 1;
        m = 0;
    }
    return (uint8_t)(sign | (uint8_t)((ef << 3) | m));
}

/* ---------------------------------------------------------------- layout */

/*
 * Routing counts, offsets and per-pair placements (sections "Send and receive buffers"
 * and "Dispatch and combine": per-expert token counts, their cumulative sums as send
 * offsets, and the offsets each receiver needs for dispatch and combine).
 *
 * idx      [N][T][R]  expert of pair (s,t,k)
 * cnt      [N][E]     cnt[s][e]  = #{(t,k) : idx[s][t][k] == e}
 * C        [N][N]     C[s][d]    = sum over d's experts of cnt[s][.]
 * soff     [N][E]     soff[s][e] = sum_{e' < e} cnt[s][e']
 * roff     [N][N]     roff[d][s] = sum_{s' < s} C[s'][d]
 * rtot     [N]        rtot[d]    = sum_s C[s][d]
 * ecnt     [N][L]     ecnt[d][l] = sum_s cnt[s][d*L+l]
 * eoff     [N][L][N]  eoff[d][l][s] = sum_{s' < s} cnt[s'][d*L+l]
 * pos      [N][T][R]  send row of the pair: soff[s][e] + rk, rk = number of earlier
 *                     (t',k') of rank s with the same expert
 * rrow     [N][T][R]  receive row in rank owner(e): roff[d][s] + pos - soff[s][d*L]
 * slot     [N][T][R]  row in expert l's grouped buffer: eoff[d][l][s] + rk, or -1
 *                     when that is >= cap
 * slot_src [N][L][cap] pair id (s*T+t)*R+k held by each grouped row, or -1
 * recv_src [N][RB]     pair id held by each receive row, or -1
 * Pairs whose expert id is out of range get pos = rrow = slot = -1 and are left out.
 */
uint32_t orc_layout(int N, int T, int E, int R, int cap, const int32_t *idx, int32_t *cnt,
                    int32_t *C, int32_t *soff, int32_t *roff, int32_t *rtot, int32_t *ecnt,
                    int32_t *eoff, int32_t *pos, int32_t *rrow, int32_t *slot,
                    int32_t *slot_src, int32_t *recv_src) {
    uint32_t status = 0;
    const int L = E / N;
    const int64_t TR = (int64_t)T * R;
    const int64_t RB = (int64_t)N * T * (R > L ? R : L);

    /* counts */
    for (int64_t i = 0; i < (int64_t)N * E; i++) cnt[i] = 0;
    for (int s = 0; s < N; s++)
        for (int t = 0; t < T; t++)
            for (int k = 0; k < R; k++) {
                int e = idx[(s * (int64_t)T + t) * R + k];
                if (e < 0 || e >= E) {
                    status |= ORC_BIT_EXPERT_RANGE;
                    continue;
                }
                cnt[(int64_t)s * E + e] += 1;
            }

    /* per-destination totals C[s][d] */
    for (int s = 0; s < N; s++)
        for (int d = 0; d < N; d++) {
            int32_t c = 0;
            for (int l = 0; l < L; l++) c += cnt[(int64_t)s * E + d * L + l];
            C[s * N + d] = c;
        }

    /* send offsets: exclusive scan of cnt[s][.] over experts */
    for (int s = 0; s < N; s++) {
        int32_t run = 0;
        for (int e = 0; e < E; e++) {
            soff[(int64_t)s * E + e] = run;
            run += cnt[(int64_t)s * E + e];
        }
    }

    /* receive offsets: exclusive scan of C[.][d] over source ranks */
    for (int d = 0; d < N; d++) {
        int32_t run = 0;
        for (int s = 0; s < N; s++) {
            roff[d * N + s] = run;
            run += C[s * N + d];
        }
        rtot[d] = run;
        if ((int64_t)run > RB) status |= ORC_BIT_RECV_BOUND;
    }

    /* grouped (expert-major) offsets: exclusive scan of cnt[.][e] over source ranks */
    for (int d = 0; d < N; d++)
        for (int l = 0; l < L; l++) {
            int e = d * L + l;
            int32_t run = 0;
            for (int s = 0; s < N; s++) {
                eoff[((int64_t)d * L + l) * N + s] = run;
                run += cnt[(int64_t)s * E + e];
            }
            ecnt[d * L + l] = run;
            if (run > cap) status |= ORC_BIT_CAPACITY;
        }

    /* per-pair placements, ranks taken in (t,k) order with one running counter per
     * expert and source rank */
    for (int64_t i = 0; i < (int64_t)N * L * cap; i++) slot_src[i] = -1;
    for (int64_t i = 0; i < (int64_t)N * RB; i++) recv_src[i] = -1;
    int32_t *running = (int32_t *)calloc((size_t)(E > 0 ? E : 1), sizeof(int32_t));
    for (int s = 0; s < N; s++) {
        for (int e = 0; e < E; e++) running[e] = 0;
        for (int t = 0; t < T; t++)
            for (int k = 0; k < R; k++) {
                int64_t q = ((int64_t)s * T + t) * R + k;
                int e = idx[q];
                if (e < 0 || e >= E) {
                    pos[q] = -1;
                    rrow[q] = -1;
                    slot[q] = -1;
                    continue;
                }
                int32_t rk = running[e]++;
                int d = e / L, l = e % L;
                int32_t p = soff[(int64_t)s * E + e] + rk;
                int32_t rr = roff[d * N + s] + (p - soff[(int64_t)s * E + d * L]);
                int32_t sl = eoff[((int64_t)d * L + l) * N + s] + rk;
                pos[q] = p;
                rrow[q] = rr;
                recv_src[(int64_t)d * RB + rr] = (int32_t)q;
                if (sl < cap) {
                    slot[q] = sl;
                    slot_src[((int64_t)d * L + l) * cap + sl] = (int32_t)q;
                } else {
                    slot[q] = -1;
                }
            }
    }
    free(running);
    (void)TR;
    return status;
}

/* ---------------------------------------------------------------- fp8 quantisation */

/*
 * Block-scaled fp8 dispatch payload (section "Evaluation": block-scaled fp8 dispatch).
 * x    [N][T][H] bf16 bits;  xq [N][T][B], B = H + 4*(H/128): the H e4m3 codes of the
 * row followed by its H/128 fp32 scales (little-endian).
 * Per 128-element block: amax = max |x| (fp32), scale = amax / 448 (fp32 division;
 * 1 when amax is 0), q = e4m3(x / scale) (fp32 division, RNE, saturating).
 */
void orc_quantize_fp8(int N, int T, int H, const uint16_t *x, uint8_t *xq) {
    const int nb = H / 128;
    const int64_t B = (int64_t)H + 4 * (int64_t)nb;
    for (int64_t r = 0; r < (int64_t)N * T; r++) {
        const uint16_t *xr = x + r * H;
        uint8_t *qr = xq + r * B;
        for (int b = 0; b < nb; b++) {
            float amax = 0.0f;
            for (int i = 0; i < 128; i++) {
                float v = fabsf(orc_bf16_to_f32(xr[b * 128 + i]));
                if (v > amax) amax = v;
            }
            float scale = (amax == 0.0f) ? 1.0f : amax / 448.0f;
            for (int i = 0; i < 128; i++) {
                float v = orc_bf16_to_f32(xr[b * 128 + i]);
                float y = v / scale;
                qr[b * 128 + i] = orc_e4m3_encode(y);
            }
            memcpy(qr + H + 4 * (int64_t)b, &scale, 4);
        }
    }
}

/* ---------------------------------------------------------------- dispatch */

/*
 * Dispatch send (section "Dispatch and combine": pack every token to be sent into the
 * send buffer at the offsets given by the cumulative counts; then one write per peer):
 *   send[s][pos[s][t][k]] = x[s][t]                           (pack)
 *   recv[d][roff[d][s] + j] = send[s][soff[s][d*L] + j],  j < C[s][d]   (the write)
 * x [N][T][B] rows of B bytes; send [N][T*R][B]; recv [N][RB][B].
 */
void orc_dispatch_send(int N, int T, int E, int R, int64_t B, const uint8_t *x,
                       const int32_t *pos, const int32_t *C, const int32_t *soff,
                       const int32_t *roff, uint8_t *send, uint8_t *recv) {
    const int L = E / N;
    const int64_t TR = (int64_t)T * R;
    const int64_t RB = (int64_t)N * T * (R > L ? R : L);
    for (int s = 0; s < N; s++)
        for (int t = 0; t < T; t++)
            for (int k = 0; k < R; k++) {
                int32_t p = pos[((int64_t)s * T + t) * R + k];
                if (p < 0) continue;
                memcpy(send + ((int64_t)s * TR + p) * B, x + ((int64_t)s * T + t) * B, (size_t)B);
            }
    for (int s = 0; s < N; s++)
        for (int d = 0; d < N; d++) {
            int64_t c = C[s * N + d];
            if (c == 0) continue;
            memcpy(recv + ((int64_t)d * RB + roff[d * N + s]) * B,
                   send + ((int64_t)s * TR + soff[(int64_t)s * E + d * L]) * B, (size_t)(c * B));
        }
}

/*
 * Dispatch receive (section "Dispatch and combine": shuffle tokens from the receive
 * buffer into the output tensor handed to the grouped GEMM). Rank d's receive buffer
 * holds, for each source s, cnt[s][e] rows of each of its experts e in expert order;
 * they go to rows eoff[d][l][s] .. + cnt[s][e] of expert l. Rows at or beyond cap are
 * dropped. bf16 (H8 == 0): ex [N][L][cap][B] rows copied verbatim. fp8 (H8 == H): the
 * first H bytes of a row go to exq [N][L][cap][H] and the H/128 scales to
 * exs [N][L][cap][H/128].
 */
void orc_dispatch_recv(int N, int T, int E, int R, int cap, int64_t B, int H8,
                       const uint8_t *recv, const int32_t *cnt, const int32_t *soff,
                       const int32_t *roff, const int32_t *eoff, uint8_t *ex, float *exs) {
    const int L = E / N;
    const int64_t RB = (int64_t)N * T * (R > L ? R : L);
    for (int d = 0; d < N; d++)
        for (int s = 0; s < N; s++)
            for (int l = 0; l < L; l++) {
                int e = d * L + l;
                int64_t n = cnt[(int64_t)s * E + e];
                int64_t src0 = roff[d * N + s] + soff[(int64_t)s * E + e] - soff[(int64_t)s * E + d * L];
                int64_t dst0 = eoff[((int64_t)d * L + l) * N + s];
                for (int64_t r = 0; r < n; r++) {
                    int64_t j = dst0 + r;
                    if (j >= cap) continue;
                    const uint8_t *src = recv + ((int64_t)d * RB + src0 + r) * B;
                    int64_t row = ((int64_t)d * L + l) * cap + j;
                    if (H8 == 0) {
                        memcpy(ex + row * B, src, (size_t)B);
                    } else {
                        int64_t nb = H8 / 128;
                        memcpy(ex + row * H8, src, (size_t)H8);
                        memcpy(exs + row * nb, src + H8, (size_t)(4 * nb));
                    }
                }
            }
}

/*
 * Identity expert for the fp8 payload: y = bf16(float(decode(q)) * scale), fp32
 * product rounded once to bf16, over the valid rows j < min(ecnt, cap) of every expert.
 */
void orc_expert_dequant(int N, int L, int cap, int H, const int32_t *ecnt, const uint8_t *exq,
                        const float *exs, uint16_t *ey) {
    const int nb = H / 128;
    for (int d = 0; d < N; d++)
        for (int l = 0; l < L; l++) {
            int n = ecnt[d * L + l];
            if (n > cap) n = cap;
            for (int j = 0; j < n; j++) {
                int64_t row = ((int64_t)d * L + l) * cap + j;
                for (int h = 0; h < H; h++) {
                    float qv = (float)orc_e4m3_decode(exq[row * H + h]);
                    float sc = exs[row * nb + h / 128];
                    float y = qv * sc;
                    ey[row * H + h] = orc_f32_to_bf16(y);
                }
            }
        }
}

/* ---------------------------------------------------------------- combine */

/*
 * Combine send (section "Dispatch and combine": the routing is already known, so tokens
 * go back with a single write per peer). First the reverse of the dispatch receive
 * shuffle puts expert outputs back into receive order in csend [N][RB][H]; then each
 * rank d writes the slice of source s back into s's crecv [N][T*R][H] at the rows its
 * dispatch send used:
 *   csend[d][roff[d][s] + soff[s][e] - soff[s][d*L] + r] = ey[d][l][eoff[d][l][s] + r]
 *   crecv[s][soff[s][d*L] + j] = csend[d][roff[d][s] + j],  j < C[s][d]
 * Rows whose grouped slot is at or beyond cap are left untouched.
 */
void orc_combine_send(int N, int T, int E, int R, int cap, int H, const uint16_t *ey,
                      const int32_t *cnt, const int32_t *C, const int32_t *soff,
                      const int32_t *roff, const int32_t *eoff, uint16_t *csend,
                      uint16_t *crecv) {
    const int L = E / N;
    const int64_t TR = (int64_t)T * R;
    const int64_t RB = (int64_t)N * T * (R > L ? R : L);
    const size_t rowb = (size_t)H * 2;
    for (int d = 0; d < N; d++)
        for (int s = 0; s < N; s++)
            for (int l = 0; l < L; l++) {
                int e = d * L + l;
                int64_t n = cnt[(int64_t)s * E + e];
                int64_t dst0 = roff[d * N + s] + soff[(int64_t)s * E + e] - soff[(int64_t)s * E + d * L];
                int64_t src0 = eoff[((int64_t)d * L + l) * N + s];
                for (int64_t r = 0; r < n; r++) {
                    int64_t j = src0 + r;
                    if (j >= cap) continue;
                    memcpy(csend + ((int64_t)d * RB + dst0 + r) * H, ey + (((int64_t)d * L + l) * cap + j) * H, rowb);
                }
            }
    for (int s = 0; s < N; s++)
        for (int d = 0; d < N; d++) {
            int64_t c = C[s * N + d];
            if (c == 0) continue;
            memcpy(crecv + ((int64_t)s * TR + soff[(int64_t)s * E + d * L]) * H,
                   csend + ((int64_t)d * RB + roff[d * N + s]) * H, (size_t)c * rowb);
        }
}

/*
 * Combine receive (section "Dispatch and combine": accumulate the tokens from the
 * receive buffer into the output tensor; the sum happens on the receiving side only):
 *   out[s][t] = bf16( sum_k w[s][t][k] * y_k ),  y_k = crecv[s][pos[s][t][k]]
 * in fp32, k ascending, multiply and add rounded separately; pairs with pos < 0 or
 * slot < 0 contribute nothing. out64 receives the same sum in fp64 (every product of an
 * fp32 weight and a bf16 value is exact in fp64).
 */
void orc_combine_recv(int N, int T, int R, int H, const uint16_t *crecv, const float *w,
                      const int32_t *pos, const int32_t *slot, uint16_t *out, double *out64) {
    const int64_t TR = (int64_t)T * R;
    for (int s = 0; s < N; s++)
        for (int t = 0; t < T; t++)
            for (int h = 0; h < H; h++) {
                float acc = 0.0f;
                double acc64 = 0.0;
                for (int k = 0; k < R; k++) {
                    int64_t q = ((int64_t)s * T + t) * R + k;
                    if (pos[q] < 0 || slot[q] < 0) continue;
                    float y = orc_bf16_to_f32(crecv[((int64_t)s * TR + pos[q]) * H + h]);
                    float prod = w[q] * y;
                    acc = acc + prod;
                    acc64 = acc64 + (double)w[q] * (double)y;
                }
                out[((int64_t)s * T + t) * H + h] = orc_f32_to_bf16(acc);
                if (out64) out64[((int64_t)s * T + t) * H + h] = acc64;
            }
}

/* ---------------------------------------------------------------- combine with partial sums */

/*
 * Combine with the weighted sum started on the expert side (section "Evaluation": DeepEP
 * accumulates on the sender side to send less data, possibly at some accuracy cost).
 * Reading: for token (s,t) the kept pairs (slot >= 0) are grouped by destination rank
 * d = e / L; the groups are numbered j = 0, 1, ... in ascending d. Group j's partial
 *   cpart[s][t][j] = bf16( sum_{k in group, k ascending} w[s][t][k] * y_k ),
 *   y_k = ey[d][e % L][slot[s][t][k]],
 * fp32 with multiply and add rounded separately; rows j >= number of groups are untouched.
 * cpart [N][T][J][H] with J = min(R, N).
 */
void orc_combine_partial_send(int N, int T, int E, int R, int cap, int H, const uint16_t *ey,
                              const float *w, const int32_t *idx, const int32_t *slot,
                              uint16_t *cpart) {
    const int L = E / N;
    const int J = R < N ? R : N;
    float *acc = (float *)malloc(sizeof(float) * (size_t)H);
    for (int s = 0; s < N; s++)
        for (int t = 0; t < T; t++) {
            int64_t q0 = ((int64_t)s * T + t) * R;
            int j = 0;
            for (int d = 0; d < N; d++) {
                int any = 0;
                for (int h = 0; h < H; h++) acc[h] = 0.0f;
                for (int k = 0; k < R; k++) {
                    int e = idx[q0 + k];
                    if (e < 0 || e >= E || slot[q0 + k] < 0 || e / L != d) continue;
                    any = 1;
                    const uint16_t *y = ey + (((int64_t)d * L + e % L) * cap + slot[q0 + k]) * H;
                    for (int h = 0; h < H; h++) {
                        float prod = w[q0 + k] * orc_bf16_to_f32(y[h]);
                        acc[h] = acc[h] + prod;
                    }
                }
                if (!any) continue;
                uint16_t *row = cpart + (((int64_t)s * T + t) * J + j) * H;
                for (int h = 0; h < H; h++) row[h] = orc_f32_to_bf16(acc[h]);
                j++;
            }
        }
    free(acc);
}

/* out[s][t] = bf16( sum_{j < groups(s,t), j ascending} float(cpart[s][t][j]) ), fp32. */
void orc_combine_partial_recv(int N, int T, int E, int R, const int32_t *idx, const int32_t *slot,
                              int H, const uint16_t *cpart, uint16_t *out) {
    const int L = E / N;
    const int J = R < N ? R : N;
    for (int s = 0; s < N; s++)
        for (int t = 0; t < T; t++) {
            int64_t q0 = ((int64_t)s * T + t) * R;
            int groups = 0;
            for (int d = 0; d < N; d++) {
                int any = 0;
                for (int k = 0; k < R; k++) {
                    int e = idx[q0 + k];
                    if (e >= 0 && e < E && slot[q0 + k] >= 0 && e / L == d) any = 1;
                }
                groups += any;
            }
            for (int h = 0; h < H; h++) {
                float acc = 0.0f;
                for (int j = 0; j < groups; j++)
                    acc = acc + orc_bf16_to_f32(cpart[(((int64_t)s * T + t) * J + j) * H + h]);
                out[((int64_t)s * T + t) * H + h] = orc_f32_to_bf16(acc);
            }
        }
}
