/*
 * moe_ep.h — C ABI of the GB300 (sm_103a) MoE expert-parallel dispatch/combine library.
 *
 * The method is the one of "Enabling trillion-parameter models on AWS EFA" (Perplexity,
 * 2025-11-04). N expert-parallel ranks each hold T tokens of hidden size H; every token
 * is routed to R of E experts, expert e living on rank owner(e) = e / L, L = E / N.
 *   dispatch: count tokens per (source rank, expert), scan the counts into collision-free
 *             contiguous offsets, pack each (token, expert) pair into the source rank's
 *             send buffer, write each destination's slice into that rank's receive buffer,
 *             and shuffle the received rows into per-expert grouped rows [L, cap, H];
 *   combine:  send expert outputs back with one write per peer and take, per token, the
 *             fp32 weighted sum of its R expert outputs, stored as bf16.
 * On one GPU all N simulated ranks live in one HBM: a rank is an address range of each
 * buffer, and a peer "RDMA write" is a device copy into the peer's receive region.
 *
 * Conventions for every entry point:
 *  - Pointers named d_* are DEVICE pointers, h_* HOST pointers. Every device buffer must be
 *    16-byte aligned; MOE_ERR_INVALID_ARG otherwise.
 *  - The caller allocates and owns all memory. The library never allocates or frees memory
 *    and never synchronises, except moe_status_sync; the batched passes (moe_forward,
 *    moe_dispatch, moe_combine, moe_forward_host) create three streams of their own and a
 *    few events per device on first use and keep them until exit. `stream` is a
 *    cudaStream_t (NULL = the legacy default stream). All calls are asynchronous on that
 *    stream; a buffer may be
 *    reused once the stream has passed its consumer (the buffer-reuse barrier between
 *    dispatch and combine of the page's section "Dispatch and combine" is stream order).
 *  - Host-checkable argument errors return MOE_ERR_INVALID_ARG before anything is launched.
 *    Data-dependent errors (bad expert id, expert capacity exceeded) never trap: kernels
 *    skip the affected pairs and OR a bit into a sticky device status word that
 *    moe_status_sync reads and clears. A failed launch returns MOE_ERR_CUDA.
 *  - Row layouts are row-major and dense; simulated rank r's part of every [N, ...] buffer
 *    starts at r * (product of the remaining dimensions).
 */
#ifndef MOE_EP_H_
#define MOE_EP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* bad dims, NULL or misaligned pointer, workspace too small */
    MOE_ERR_EXPERT_RANGE = 2, /* an expert id outside [0, E); its pair was left out */
    MOE_ERR_CAPACITY = 3,     /* an expert got more than cap pairs; the excess was dropped */
    MOE_ERR_RECV_BOUND = 4,   /* a rank received more than N*T*max(R,E/N) rows (cannot
                                 happen with in-range ids; checked defensively) */
    MOE_ERR_CUDA = 5,         /* a CUDA call or launch failed */
    MOE_ERR_TIMEOUT = 6       /* a bounded wait inside a kernel ran out; work was skipped */
} moe_status;

typedef enum {
    MOE_PAYLOAD_BF16 = 0,          /* rows of H bf16 values, B = 2H bytes */
    MOE_PAYLOAD_FP8_E4M3_B128 = 1  /* rows of H e4m3 codes then H/128 fp32 scales,
                                      B = H + 4*(H/128) bytes (section "Evaluation":
                                      block-scaled fp8 dispatch, bf16 combine) */
} moe_payload;

/* Problem size, in the page's notation (section "Send and receive buffers": N ranks each
 * dispatch T tokens, each routed to R of E experts). */
typedef struct {
    int32_t N;       /* simulated expert-parallel ranks, >= 1 */
    int32_t T;       /* tokens per rank, >= 0 */
    int32_t H;       /* hidden size: multiple of 8 (bf16), of 128 (fp8) */
    int32_t E;       /* experts in total, multiple of N; E/N local experts per rank */
    int32_t R;       /* experts per token, >= 1 */
    int32_t cap;     /* rows per expert in the grouped buffers; 0 means N*T */
    int32_t payload; /* moe_payload of the dispatched rows */
} moe_dims;

/* Kernel ids reported through moe_prof_t. */
typedef enum {
    MOE_K_ROUTE_COUNT = 0,     /* routing-count histogram per 256-pair chunk + stable ranks */
    MOE_K_LAYOUT_MAPS = 1,     /* per-pair placements and inverse maps */
    MOE_K_QUANT_FP8 = 2,       /* block-scaled fp8 quantisation */
    MOE_K_PACK = 3,            /* dispatch send: token rows -> send rows */
    MOE_K_SCATTER = 4,         /* dispatch "RDMA write": send slices -> peers' receive rows */
    MOE_K_UNPACK = 5,          /* dispatch recv: receive rows -> grouped expert rows */
    MOE_K_EXPERT = 6,          /* identity expert (fp8 dequantisation or bf16 copy) */
    MOE_K_COMBINE_PACK = 7,    /* combine send: grouped rows -> receive order */
    MOE_K_COMBINE_SCATTER = 8, /* combine "RDMA write": back to the source ranks */
    MOE_K_COMBINE_REDUCE = 9,  /* combine recv: weighted sum over R -> bf16 */
    MOE_K_ROUTE_SCAN = 10,     /* per-rank totals and every exclusive scan */
    MOE_K_PACK_PUSH = 11,      /* direct push: token rows -> owners' receive rows */
    MOE_K_COMBINE_PUSH = 12,   /* direct push: grouped rows -> sources' combine rows */
    MOE_K_COMBINE_PARTIAL = 13, /* expert-side partial sums, one row per (token, rank) */
    MOE_K_COMBINE_SUM = 14,    /* source-side sum of the partial rows -> bf16 */
    MOE_K_DISPATCH_SPLIT = 15, /* split-phase dispatch: push, signal, wait, shuffle in one launch */
    MOE_K_QUANT_PACK = 16,     /* fp8 quantisation fused into the pack */
    MOE_K_DISPATCH_DEDICATED = 17, /* split-phase dispatch with dedicated space and piggybacked routing */
    MOE_K_DISPATCH_FUSED = 18, /* pack, write and shuffle in one kernel (bf16) */
    MOE_K_QUANT_DISPATCH_FUSED = 19, /* fp8 quantisation, pack, write and shuffle in one kernel */
    MOE_K_COMBINE_FUSED = 20,  /* combine pack, write and weighted sum in one kernel */
    MOE_K_NUM = 21
} moe_kernel_id;

/* Optional per-kernel timing. When moe_layout_t.prof is non-NULL, every kernel the library
 * launches is bracketed by cudaEventRecord(events[2n]) and cudaEventRecord(events[2n+1]) on
 * the call's stream, kernel[n] receives its moe_kernel_id and n is incremented, until n
 * reaches MOE_PROF_MAX. The caller creates the events (cudaEvent_t cast to void*) and
 * resets n.
 * Cold timing: when `flush` is non-NULL (a device buffer of flush_bytes, a multiple of 16
 * and best at least twice the L2 size), a kernel of the library reads the whole buffer on
 * the stream before each bracketed launch's first event, so every timed kernel starts with
 * the previous kernels' rows evicted from L2 (their dirty lines written back during the
 * read, outside the bracket). The read kernel is not bracketed; it writes at most 16 bytes
 * at the start of the buffer. flush_bytes below 16 or not a multiple of 16 turns it off. */
#define MOE_PROF_MAX 32
typedef struct {
    void *events[2 * MOE_PROF_MAX];
    int32_t kernel[MOE_PROF_MAX];
    int32_t n;
    void *flush;
    size_t flush_bytes;
} moe_prof_t;

/* moe_layout_t.flags */
/* Row movers. By default each launch picks one: TMA bulk copies for the one-to-one moves
 * when every issuer warp has at least 40 rows to stream, 16-byte register loads/stores for
 * pack (one row to R destinations) and for smaller problems. Rows that are not 16-byte
 * multiples (fp8 with H % 512 != 0) always take the register path. */
#define MOE_FLAG_LDG_MOVER 0x1u /* force the register mover for every move */
#define MOE_FLAG_TMA_MOVER 0x4u /* force the TMA mover wherever rows allow it */
/* Direct push: the send halves write straight into the destination's buffer, the way the
 * page's intra-node path pushes tokens over NVLink into peers' mapped receive buffers
 * (sections "MoE all-to-all over EFA" and "Dispatch and combine"). moe_dispatch_send packs
 * each pair into its owner's receive row (d_send is not used and may be NULL), and
 * moe_combine_send writes each expert output into its source's combine row (d_csend is
 * not used and may be NULL). The receive, grouped and combine buffers hold exactly what
 * they hold without the flag; the per-peer write step is fused away. */
#define MOE_FLAG_DIRECT_PUSH 0x8u
/* fp8 payload in moe_forward: quantise into d_xq with moe_quantize_fp8_b128 and dispatch
 * those rows (two kernels), instead of the default moe_quantize_dispatch_send, which
 * quantises inside the pack and leaves d_xq unwritten. Same receive and grouped contents. */
#define MOE_FLAG_STAGED_QUANT 0x10u
/* moe_forward_host with device-accessible host buffers: run the kernels on the host memory
 * itself (the pack reads the tokens and the reduce writes the output over the host link)
 * instead of the default copy-engine pipeline. */
#define MOE_FLAG_HOST_MAPPED 0x20u
/* moe_forward and moe_forward_host: run the pass as one token batch on the caller's stream
 * (for moe_forward_host: copies, then the pass, then the copy back; or, with
 * MOE_FLAG_HOST_MAPPED, the pass alone) instead of the default token batches. */
#define MOE_FLAG_ONE_BATCH 0x40u
/* The whole-pass and whole-phase calls (moe_forward, moe_dispatch, moe_combine and the
 * copy-engine pipeline of moe_forward_host) run each phase of a token batch as one kernel:
 * dispatch reads (and, for fp8, quantises) each token row once and stores it to its send
 * rows, the owners' receive rows and the grouped rows; combine reads each kept pair's expert
 * output row once, stores it to its receive-order row and its source's combine row, and sums
 * the token's rows into its output. Every buffer ends up as with the separate calls, byte for
 * byte, and so does the output. With MOE_FLAG_DIRECT_PUSH the same two kernels write no send
 * rows and no receive-order rows, as the direct-push calls do not. This flag runs the phases as
 * the separate calls do instead (pack, write, shuffle; combine pack, write, sum). */
#define MOE_FLAG_SEPARATE_MOVES 0x80u
#define MOE_FLAG_NO_PDL 0x2u    /* launch without programmatic dependent launch (by default
                                   each kernel may be scheduled while its predecessor in the
                                   stream drains; it waits for it before touching memory) */

/*
 * Routing layout. Device arrays carved by moe_layout_init from one caller workspace, filled
 * by moe_layout, read by every later call (section "Send and receive buffers": per-expert
 * counts are exchanged first, so every rank knows where its writes go and at which offset
 * it receives from each rank; section "Dispatch and combine": the receiver computes the
 * offsets needed for dispatch and combine). int32, row-major:
 *   cnt  [N][E]   tokens rank s routes to expert e
 *   C    [N][N]   C[s][d]: rows rank s sends to rank d
 *   soff [N][E]   exclusive scan of cnt[s][.] over e: send offsets
 *   roff [N][N]   roff[d][s]: exclusive scan of C[.][d] over s: receive offsets
 *   rtot [N]      rows rank d receives (<= N*T*max(R,E/N))
 *   ecnt [N][L]   rows expert l of rank d receives
 *   eoff [N][L][N] eoff[d][l][s]: exclusive scan of cnt[.][d*L+l] over s
 *   pos  [N][T][R] send row of pair (s,t,k): soff[s][e] + rk, rk = number of earlier
 *                  (t',k') of rank s with the same expert; -1 for a bad expert id
 *   rrow [N][T][R] receive row of the pair in rank owner(e); -1 for a bad id
 *   slot [N][T][R] grouped row of the pair in expert e: eoff[d][l][s] + rk; -1 if >= cap
 *   slot_src [N][L][cap] pair id (s*T+t)*R+k of each grouped row, -1 if unused
 *   recv_src [N][RB]     pair id of each receive row, -1 if unused (RB = N*T*max(R,E/N))
 *   gsend [N*T*R]  global send row of each pair, s*T*R + pos (row of d_send), or -1
 *   grecv [N*T*R]  global receive row, owner(e)*RB + rrow (row of d_recv), or -1
 *   gslot [N*T*R]  global grouped row, e*cap + slot (row of d_expert_x), or -1 when the
 *                  pair's expert id is bad or the pair was dropped for capacity
 *   status   [1]         sticky error bits, bit (1 << moe_status)
 *   scratch  internal: per-chunk counts [N][ceil(T*R/256)][E], per-rank counters [N],
 *            per-token group counts of the partial combine [N][T] and the split-phase
 *            arrival counters [max(N, 32)][N] (+ 2)
 * Host-side fields (set by the caller after moe_layout_init, read at each call):
 *   flags, prof, tma_stages (0 = automatic, else 1..32 stages per TMA mover CTA),
 *   ctas_per_sm (0 = automatic, else mover CTAs per SM), batches (token batches of
 *   moe_forward's micro-batches, of moe_dispatch / moe_combine and of moe_dispatch_split
 *   (0 = automatic, else 1..32) and of moe_forward_host's copy-engine pipeline (0 =
 *   automatic, else 1..24); see moe_batches), win_lo / win_hi (the rank window, below).
 *
 * Rank window (expert parallelism over several GPUs, one process each; section "Send and
 * receive buffers": every rank knows where its writes go and where it receives from each
 * rank; section "MoE all-to-all over EFA": one write per peer). With win_hi > 0 the layout
 * describes all N ranks (moe_layout reads the routing of every rank, d_idx [N][T][R]) but the
 * data entry points below work on the ranks [win_lo, win_hi) only, whose buffers are
 * window-local: rank win_lo + i is row block i of every [N, ...] buffer, which holds
 * n = win_hi - win_lo blocks (d_x [n][T][H], d_send [n][T*R][B], d_recv [n][RB][B],
 * d_expert_x [n][L][cap][...], d_csend [n][RB][H], d_crecv [n][T*R][H], d_w [n][T][R],
 * d_out [n][T][H]). Within the window:
 *   moe_dispatch_send / moe_quantize_dispatch_send pack the window's tokens and write the
 *     slices whose destination is in the window (the slices to other ranks stay in d_send
 *     for the caller to move, at the rows moe_exchange_plan lists);
 *   moe_dispatch_recv shuffles the receive rows of the window's ranks (the slices from
 *     other ranks must have been written into d_recv first);
 *   moe_expert_identity works on the window's experts;
 *   moe_combine_send writes the window's expert outputs in receive order and writes back
 *     the slices whose source is in the window (the others stay in d_csend for the caller);
 *   moe_combine_recv sums the window's tokens (the slices from other ranks must have been
 *     written into d_crecv first).
 * moe_quantize_fp8_b128 quantises the window's token rows. Every other data entry point, and
 * MOE_FLAG_DIRECT_PUSH, needs the whole group (win_lo = win_hi = 0, or 0 and N): otherwise
 * MOE_ERR_INVALID_ARG. A window runs each call as one token batch.
 */
typedef struct {
    int32_t *cnt, *C, *soff, *roff, *rtot, *ecnt, *eoff;
    int32_t *pos, *rrow, *slot, *slot_src, *recv_src;
    int32_t *gsend, *grecv, *gslot;
    int32_t *status;
    int32_t *scratch; /* internal: chunk count table of the routing-count kernels */
    uint32_t flags;
    moe_prof_t *prof;
    int32_t tma_stages;
    int32_t ctas_per_sm;
    int32_t batches;
    int32_t win_lo, win_hi; /* rank window [win_lo, win_hi); 0, 0: all N ranks */
} moe_layout_t;

/* Device buffers of one whole pass (moe_forward). Shapes, with B = row bytes,
 * RB = N*T*max(R,E/N), L = E/N:
 *   x        [N][T][H]  bf16 tokens (input)
 *   xq       [N][T][B]  fp8 rows (fp8 payload only; written by the pass)
 *   idx      [N][T][R]  int32 expert ids (input)
 *   w        [N][T][R]  fp32 router weights (input)
 *   send     [N][T*R][B]
 *   recv     [N][RB][B]
 *   expert_x [N][L][cap][B] (bf16) or [N][L][cap][H] e4m3 codes (fp8)
 *   expert_scale [N][L][cap][H/128] fp32 (fp8 only, else NULL)
 *   expert_y [N][L][cap][H] bf16; for bf16 it may equal expert_x (identity by aliasing)
 *   csend    [N][RB][H] bf16 (may alias recv when B == 2H)
 *   crecv    [N][T*R][H] bf16 (may alias send when B == 2H)
 *   out      [N][T][H]  bf16 (output) */
typedef struct {
    uint16_t *x;
    uint8_t *xq;
    int32_t *idx;
    float *w;
    void *send;
    void *recv;
    void *expert_x;
    float *expert_scale;
    uint16_t *expert_y;
    uint16_t *csend;
    uint16_t *crecv;
    uint16_t *out;
} moe_buffers_t;

/* Validates dims: N >= 1, T >= 0, E % N == 0, R >= 1, cap >= 0, H % 8 == 0 (bf16) or
 * H % 128 == 0 (fp8), and the library's limits (E <= 1536, N <= 2048, all row
 * counts below 2^31). MOE_OK or MOE_ERR_INVALID_ARG. */
moe_status moe_check_dims(const moe_dims *dims);

/* N*T*max(R, E/N): the receive rows one rank can need (section "Send and receive
 * buffers": with all tokens routed to one rank, it receives at most N*T*max(R,E/N)). */
size_t moe_recv_capacity_rows(const moe_dims *dims);

/* Bytes per dispatched row: 2H (bf16) or H + 4*(H/128) (fp8). 0 for invalid dims. */
size_t moe_row_bytes(const moe_dims *dims);

/* Effective per-expert capacity (cap, or N*T when cap is 0). */
int32_t moe_capacity(const moe_dims *dims);

/* Bytes of device workspace moe_layout_init needs (every array above, 256-byte aligned). */
size_t moe_layout_workspace_bytes(const moe_dims *dims);

/* Carves the layout arrays out of d_ws (ws_bytes >= moe_layout_workspace_bytes) into *out,
 * zeroes the status word and the internal counter on `stream`, and sets the host-side
 * fields to their defaults (flags 0, prof NULL, automatic tuning). */
moe_status moe_layout_init(const moe_dims *dims, void *d_ws, size_t ws_bytes, moe_layout_t *out,
                           void *stream);

/* Dispatch-send step 1-2 and the receiver's offsets (section "Dispatch and combine":
 * aggregate the routing in shared memory into per-expert token counts, then their
 * cumulative sums as send offsets; the receiver centralises all ranks' routing and
 * computes the offsets for dispatch and combine). Reads d_idx [N][T][R] int32, fills every
 * array of *lay. Three kernels: per-chunk counts and ranks (the last CTA of each source
 * rank sums its chunks), the scans, the per-pair maps. */
moe_status moe_layout(const moe_dims *dims, const int32_t *d_idx, const moe_layout_t *lay, void *stream);

/* Block-scaled fp8 quantisation of the dispatch payload (section "Evaluation"): for each
 * 128-element block of each token row of d_x [N][T][H] bf16, scale = amax/448 (1 if amax is
 * 0) and q = e4m3(x/scale), round to nearest even, saturating. Writes d_xq [N][T][B]: the
 * H codes of a row, then its H/128 fp32 scales. dims->payload must be fp8. */
moe_status moe_quantize_fp8_b128(const moe_dims *dims, const uint16_t *d_x, uint8_t *d_xq,
                                 const moe_layout_t *lay, void *stream);

/* Dispatch send (section "Dispatch and combine": pack every token into the send buffer at
 * its offsets; then one write per peer, the TransferEngine "scatter" of section "MoE
 * routing with TransferEngine"): send[s][pos[s][t][k]] = x[s][t], then
 * recv[d][roff[d][s] + j] = send[s][soff[s][d*L] + j] for j < C[s][d].
 * d_x [N][T][B] (bf16 tokens, or fp8 rows from moe_quantize_fp8_b128), d_send [N][T*R][B],
 * d_recv [N][RB][B]. Receive rows at or beyond rtot[d] are not written. Two kernels (one
 * with MOE_FLAG_DIRECT_PUSH). */
moe_status moe_dispatch_send(const moe_dims *dims, const moe_layout_t *lay, const void *d_x, void *d_send,
                             void *d_recv, void *stream);

/* Quantisation fused into dispatch send (section "Evaluation": block-scaled fp8 dispatch;
 * section "Dispatch and combine": the sender packs tokens for single writes per peer):
 * for an fp8 payload, each bf16 token row of d_x [N][T][H] is quantised once in registers
 * (the rule of moe_quantize_fp8_b128) and its B-byte fp8 row written to the send rows of
 * its pairs, then scattered as by moe_dispatch_send; with MOE_FLAG_DIRECT_PUSH it is
 * written straight into the owners' receive rows (d_send unused, may be NULL). d_recv
 * ends up byte-identical to moe_quantize_fp8_b128 followed by moe_dispatch_send; no
 * quantised copy of d_x is kept. A bf16 payload is MOE_ERR_INVALID_ARG. */
moe_status moe_quantize_dispatch_send(const moe_dims *dims, const moe_layout_t *lay, const uint16_t *d_x,
                                      void *d_send, void *d_recv, void *stream);

/* Dispatch send that allocates nothing, for callers that cannot call cudaMalloc (code
 * under a fixed memory plan made before serving, allocator hooks that must not re-enter the
 * allocator, hosts that only pass in tensors they already own). The page has no counterpart:
 * it is an interface variant of moe_dispatch_send, with the same results in d_recv, whose
 * send buffer lives in a file-scope device array of the library (64 MiB) instead of a
 * caller buffer. Arguments are those of moe_dispatch_send without d_send.
 *  - Sizes: N*T*R*B must be at most 64 MiB (B = row bytes), else MOE_ERR_INVALID_ARG.
 *  - The first call on a device looks the array's address up (cudaGetSymbolAddress) with
 *    that device current; make that first call before any stream capture. The address is
 *    the one of the device's primary context: do not call this after cudaDeviceReset or with
 *    another context of the device current.
 *  - MOE_FLAG_DIRECT_PUSH is ignored: the rows are always packed into the array, then
 *    scattered (moe_dispatch_send with that flag needs no send buffer at all).
 *  - The array is shared by every call and keeps the last call's rows; calls that overlap
 *    on the GPU (other streams or threads) race on it. Every GPU that loads the library
 *    holds the 64 MiB until the process exits.
 *  - Calls no allocating routine (no cudaMalloc, cudaFree or library allocator). */
moe_status moe_dispatch_send_noalloc(const moe_dims *dims, const moe_layout_t *lay, const void *d_x,
                                     void *d_recv, void *stream);

/* Split-phase dispatch (section "Dispatch and combine": dispatch is split into a sender half
 * that fills the peers' buffers and signals, and a receiver half that waits for every transfer
 * of its peers and then shuffles the tokens into the grouped-GEMM input; section "MoE
 * all-to-all over EFA": inside a node the sender writes straight into the peers' buffers).
 * Results are those of moe_dispatch_send with MOE_FLAG_DIRECT_PUSH followed by
 * moe_dispatch_recv: d_recv [N][RB][B] holds every receive row, d_expert_x / d_expert_scale
 * the grouped rows (same layouts as moe_dispatch_recv).
 * One cooperative launch over nb token batches (tokens [j*T/nb, (j+1)*T/nb) of every rank;
 * nb = lay->batches if set, else about one per 32 MB of pushed rows; at most 32 and T).
 * Sender warps push each batch's
 * token rows into the owners' receive rows and, once their rows of the batch have landed,
 * signal the batch on a counter per (batch, source rank); receiver warps take the batch's
 * pairs, wait until the pair's source has signalled every token of the batch, and copy the
 * row into its expert's slot, while the batch's rows are still in L2. Each wait is bounded
 * (1 s): on expiry the status word gets the MOE_ERR_TIMEOUT bit, later waits of the call give
 * up at once, the grouped rows of unfinished batches are left unwritten, and the call still
 * completes. The counters live in the layout workspace, start at zero and are zeroed again by
 * the call; calls that share a layout must not overlap on the GPU.
 * withhold_source: failure injection for tests; source rank s's signals are never sent, so
 * the waits for its rows time out (its receive rows are still written, its grouped rows are
 * not). Pass -1 in normal use; other negative values and values >= N are
 * MOE_ERR_INVALID_ARG, and so is R > 32. */
moe_status moe_dispatch_split(const moe_dims *dims, const moe_layout_t *lay, const void *d_x, void *d_recv,
                              void *d_expert_x, float *d_expert_scale, int32_t withhold_source, void *stream);

/* Split-phase dispatch with per-sender dedicated space and the routing information
 * piggybacked on the first writes (section "Send and receive buffers": each receiver
 * reserves a small dedicated space per sender; the sender dispatches part of its tokens
 * together with the routing-information write, and after the routes are exchanged the
 * remaining tokens go with one write per peer; section "Dispatch and combine": the receiver
 * centralises its peers' routing, computes its offsets, waits for every transfer and
 * shuffles the tokens into the grouped-GEMM input).
 * Senders use only their own routing from *lay (cnt, soff, pos, filled by moe_layout);
 * receivers compute their offsets only from the counts the senders report. Buffers:
 *   d_ded  [N][N][K][B]: rank d's dedicated rows for sender s: rows j < K of the slice
 *          (d, s) (the rows s sends to d, in s's send order);
 *   d_main [N][RB][B]: rank d's shared region: rows j >= K of each slice, sender after
 *          sender (the slice of s at place sum over s' < s of max(C[s'][d] - K, 0));
 *   d_xchg moe_dedicated_exchange_bytes(dims) bytes: the reported counts, the receivers'
 *          offsets and the flags (zeroed by the call);
 *   d_expert_x / d_expert_scale: the grouped rows, as moe_dispatch_recv writes them.
 * One cooperative launch (after a memset of the flags); every wait bounded (1 s, then
 * MOE_ERR_TIMEOUT and the call still completes). K >= 0 (K = 0: no dedicated rows).
 * withhold_slice: failure injection for tests (the row signals of slice d*N + s are never
 * sent); -1 in normal use. MOE_ERR_INVALID_ARG for R > 32, K < 0 or a bad withhold_slice. */
size_t moe_dedicated_exchange_bytes(const moe_dims *dims);
moe_status moe_dispatch_dedicated(const moe_dims *dims, const moe_layout_t *lay, const int32_t *d_idx,
                                  const void *d_x, int32_t K, void *d_ded, void *d_xchg, void *d_main,
                                  void *d_expert_x, float *d_expert_scale, int32_t withhold_slice, void *stream);

/* Dispatch receive (section "Dispatch and combine": shuffle tokens from the receive buffer
 * into the tensor handed to the grouped GEMM): every receive row of rank d goes to row
 * slot of its expert l. bf16: d_expert_x [N][L][cap][H] bf16, d_expert_scale unused.
 * fp8: d_expert_x [N][L][cap][H] e4m3 codes, d_expert_scale [N][L][cap][H/128] fp32.
 * Rows j >= ecnt[d][l] are not written. One kernel. */
moe_status moe_dispatch_recv(const moe_dims *dims, const moe_layout_t *lay, const void *d_recv,
                             void *d_expert_x, float *d_expert_scale, void *stream);

/* Identity expert standing in for the grouped GEMM (not a step of the paper's kernels):
 * fp8: y = bf16(float(q) * scale) on every used grouped row; bf16: y = x, no launch when
 * d_expert_y == d_expert_x, else a copy of the used rows. d_expert_y [N][L][cap][H] bf16. */
moe_status moe_expert_identity(const moe_dims *dims, const moe_layout_t *lay, const void *d_expert_x,
                               const float *d_expert_scale, uint16_t *d_expert_y, void *stream);

/* Combine send (section "Dispatch and combine": routing is already known, tokens go back
 * with a single write per peer): the reverse receive shuffle
 * csend[d][rrow(s,t,k)] = expert_y[d][l][slot(s,t,k)], then the write back
 * crecv[s][soff[s][d*L] + j] = csend[d][roff[d][s] + j]. d_expert_y [N][L][cap][H] bf16,
 * d_csend [N][RB][H] bf16, d_crecv [N][T*R][H] bf16. Pairs dropped for capacity are
 * skipped (their crecv rows are not written). Two kernels (one with MOE_FLAG_DIRECT_PUSH). */
moe_status moe_combine_send(const moe_dims *dims, const moe_layout_t *lay, const uint16_t *d_expert_y,
                            uint16_t *d_csend, uint16_t *d_crecv, void *stream);

/* Combine receive (section "Dispatch and combine": accumulate the tokens from the receive
 * buffer into the output tensor; accumulation happens on the receiving side only, section
 * "Evaluation"): out[s][t] = bf16(sum_k w[s][t][k] * crecv[s][pos[s][t][k]]), fp32 products
 * and sums rounded separately, k ascending, dropped or invalid pairs skipped.
 * d_crecv [N][T*R][H] bf16, d_w [N][T][R] fp32, d_out [N][T][H] bf16. One kernel. */
moe_status moe_combine_recv(const moe_dims *dims, const moe_layout_t *lay, const uint16_t *d_crecv,
                            const float *d_w, uint16_t *d_out, void *stream);

/* Whole phases, as the page's dispatch and combine calls (section "Dispatch and combine"):
 * moe_dispatch leaves what moe_dispatch_send followed by moe_dispatch_recv leaves (fp8: d_x
 * holds the bf16 token rows, always quantised inside the pack as moe_quantize_dispatch_send
 * does, so MOE_FLAG_STAGED_QUANT does not apply; d_send unused with MOE_FLAG_DIRECT_PUSH);
 * moe_combine leaves what moe_combine_send followed by moe_combine_recv leaves. One kernel
 * per phase and token batch (with or without MOE_FLAG_DIRECT_PUSH) unless
 * MOE_FLAG_SEPARATE_MOVES. Arguments
 * as in those calls; the expert work goes between the two. Each phase may run in nb token batches
 * (nb = moe_batches(dims, lay, 2): lay->batches, else none up to 2048 tokens of all ranks
 * and about T/8 beyond, at most 16; one with MOE_FLAG_ONE_BATCH), batch j covering tokens
 * [j*T/nb, (j+1)*T/nb) of every rank, odd batches on the library's
 * second stream, which the caller's stream waits for before the call returns. Every
 * buffer ends up as with the separate calls, bit for bit. */
moe_status moe_dispatch(const moe_dims *dims, const moe_layout_t *lay, const void *d_x, void *d_send,
                        void *d_recv, void *d_expert_x, float *d_expert_scale, void *stream);
moe_status moe_combine(const moe_dims *dims, const moe_layout_t *lay, const uint16_t *d_expert_y,
                       uint16_t *d_csend, uint16_t *d_crecv, const float *d_w, uint16_t *d_out, void *stream);

/* Combine with the weighted sum started on the expert side (section "Evaluation": DeepEP
 * accumulates on the sender side to send less data, at some accuracy cost; this library's
 * default combine accumulates on the receiving side only, as the page's kernels do).
 * For token (s,t) the pairs kept in the grouped buffers are grouped by destination rank
 * d = owner(e), groups numbered j = 0, 1, ... in ascending d; J = min(R, N).
 *  moe_combine_send_partial: each expert rank writes, straight into the source's buffer,
 *    d_cpart[s][t][j] = bf16(sum over the group's pairs, k ascending, of w * y), fp32 with
 *    products and sums rounded separately. d_expert_y [N][L][cap][H] bf16, d_w [N][T][R]
 *    fp32, d_cpart [N][T][J][H] bf16; rows j >= the token's group count are not written.
 *  moe_combine_recv_partial: d_out[s][t] = bf16(sum over j ascending of d_cpart[s][t][j]),
 *    fp32, with the group counts the send half left in the layout's scratch: call it after
 *    moe_combine_send_partial on the same layout. Every token moves one row per group
 *    instead of one per expert. */
moe_status moe_combine_send_partial(const moe_dims *dims, const moe_layout_t *lay, const uint16_t *d_expert_y,
                                    const float *d_w, uint16_t *d_cpart, void *stream);
moe_status moe_combine_recv_partial(const moe_dims *dims, const moe_layout_t *lay, const uint16_t *d_cpart,
                                    uint16_t *d_out, void *stream);

/* One whole pass, with the results of moe_layout, moe_quantize_dispatch_send (fp8; or
 * moe_quantize_fp8_b128 + moe_dispatch_send with MOE_FLAG_STAGED_QUANT) or moe_dispatch_send
 * (bf16), moe_dispatch_recv, moe_expert_identity, moe_combine_send and moe_combine_recv in
 * every buffer, bit for bit (each phase one kernel per token batch unless
 * MOE_FLAG_SEPARATE_MOVES; staged fp8 quantisation runs those calls). Returns the first
 * error. bufs->x, idx, w and out may also be device-accessible host memory.
 * After the layout, the pass runs as nb micro-batches (nb = moe_batches(dims, lay, 0):
 * lay->batches (at most 32 and T), or automatically about one per 55 MB of dispatch and
 * combine rows (N*T*R pairs x (row bytes + 2H)), rounded up to an even count from 3, at most
 * 20 and T (fp8 rows, MOE_FLAG_DIRECT_PUSH or MOE_FLAG_SEPARATE_MOVES: one per 60 MB, at
 * most 16);
 * one with MOE_FLAG_ONE_BATCH or staged fp8 quantisation). Micro-batch j covers tokens
 * [j*T/nb, (j+1)*T/nb) of every rank and runs the dispatch, the identity expert and the
 * combine on only those tokens' rows (the same kernels, restricted to a token range), odd
 * micro-batches on the library's second stream (created on first use, kept until exit);
 * the caller's stream waits for it before the call returns. Every buffer ends up as in one
 * batch, bit for bit.
 * Graph capture: a captured call forks the library's stream into the capture and joins it
 * back, so the pass captures like any other stream work; while a capture that holds such
 * a call is open on a device, no other thread may run a multi-batch moe_forward or
 * moe_forward_host on that device (its work would land in the open capture). */
moe_status moe_forward(const moe_dims *dims, const moe_layout_t *lay, const moe_buffers_t *bufs, void *stream);

/* moe_forward with host inputs h_x [N][T][H] bf16, h_idx [N][T][R], h_w [N][T][R] and host
 * output h_out [N][T][H] (pinned for the copies to be asynchronous; pageable works too).
 * Default: a pipeline over nb token batches (tokens [j*T/nb, (j+1)*T/nb) of every rank;
 * nb = lay->batches, or automatically about 2 sqrt(token-row MB), at most 24 and T).
 * A copy-engine stream of the library copies h_idx and h_w into bufs->idx/w, then each
 * batch's token rows into bufs->x; the caller's stream runs the layout as soon as idx is
 * there, then each batch's dispatch, identity expert and combine once its rows are there;
 * a second copy-engine stream copies each finished batch's rows of bufs->out into h_out.
 * The copies of one batch overlap the device work of the others without taking SMs from
 * it. When an average batch's combine rows (pairs x 2H bytes) take at most 40% of the L2,
 * odd batches' device work runs on the library's second stream; otherwise all of it
 * runs on `stream` and the first and last batches are half the size of the others. The
 * streams and their events are created on the first such call per device and kept until
 * exit; the caller's stream waits for them before the call returns, so `stream` orders
 * everything as usual (and the pass can be captured into a CUDA graph).
 * With MOE_FLAG_ONE_BATCH (or fp8 with MOE_FLAG_STAGED_QUANT): copies in, moe_forward in one
 * batch, copy out, all on `stream`.
 * With MOE_FLAG_HOST_MAPPED and all four buffers pinned memory the device can address
 * (cudaHostAlloc / cudaHostRegister; over NVLink-C2C on Grace-Blackwell), the kernels read
 * the inputs and write the output there directly and bufs->x/idx/w/out are not used; with
 * T >= 2 (and neither direct push, staged fp8 quantisation nor MOE_FLAG_ONE_BATCH)
 * that pass runs in two token batches, the library's second stream taking the
 * scatter and unpack of the first batch and its reduce while the caller's stream packs and
 * sends the second (otherwise it is moe_forward on the mapped memory). Asynchronous: the
 * caller synchronises `stream` before reading h_out. */
moe_status moe_forward_host(const moe_dims *dims, const moe_layout_t *lay, const moe_buffers_t *bufs,
                            const uint16_t *h_x, const int32_t *h_idx, const float *h_w, uint16_t *h_out,
                            void *stream);

/* The slices a rank window sends to or receives from the ranks outside it (section "Send
 * and receive buffers": with the counts known, each rank writes one contiguous slice per
 * peer at offsets both sides derive from them). The N ranks are split into nwin windows,
 * window w holding ranks [h_bounds[w], h_bounds[w+1]) (h_bounds ascending, h_bounds[0] = 0,
 * h_bounds[nwin] = N); `me` is the caller's window. h_C [N][N], h_soff [N][E] and
 * h_roff [N][N] are host copies of the layout's arrays.
 *  direction 0 (dispatch): sending = 1 lists, for every source s in the window and
 *    destination d outside it with C[s][d] > 0, the rows of d_send (window-local row
 *    (s - lo)*T*R + soff[s][d*L]); sending = 0 lists, for every destination d in the window
 *    and source s outside it, the rows of d_recv ((d - lo)*RB + roff[d][s]).
 *  direction 1 (combine): sending = 1 lists the rows of d_csend that go back to sources
 *    outside the window ((d - lo)*RB + roff[d][s], d in the window); sending = 0 lists the
 *    rows of d_crecv that arrive from them ((s - lo)*T*R + soff[s][d*L], s in the window).
 * Each slice is C[s][d] rows; `peer` is the window on the other side. Slices are listed in
 * ascending (s, d) order, so the k-th slice window p sends to window q is the k-th slice q
 * receives from p. Writes at most max_out slices to out (may be NULL) and returns how many
 * there are, or -1 for bad arguments. Host only, no CUDA call. */
typedef struct {
    int32_t peer;       /* the other window */
    int32_t s, d;       /* source and destination rank of the slice */
    int32_t rows;       /* C[s][d] */
    int64_t local_row;  /* first row in the caller's window-local buffer */
} moe_slice_t;
int64_t moe_exchange_plan(const moe_dims *dims, const int32_t *h_C, const int32_t *h_soff, const int32_t *h_roff,
                          int32_t nwin, const int32_t *h_bounds, int32_t me, int32_t direction, int32_t sending,
                          moe_slice_t *out, int64_t max_out);

/* Token batches for these dims and layout settings (lay->batches, lay->flags): which = 0:
 * moe_forward's micro-batches; 1: moe_forward_host's copy-engine pipeline; 2: the phases of
 * moe_dispatch and moe_combine. 1 means one batch; 0 for bad arguments. Host only, no CUDA
 * call. */
int32_t moe_batches(const moe_dims *dims, const moe_layout_t *lay, int32_t which);

/* Synchronises `stream`, reads and clears the device status word. Returns MOE_OK or the
 * lowest-numbered error whose bit is set; *bits_out (may be NULL) receives all bits. */
moe_status moe_status_sync(const moe_layout_t *lay, void *stream, uint32_t *bits_out);

/* Static string for a status code. */
const char *moe_status_string(moe_status s);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_EP_H_ */
