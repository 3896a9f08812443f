// Internal interface between the host side (validation, plans, launches) and the kernels of the gx_gemm library.
// Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sdmgx {

// Bits of the device error word (one 32-bit word per device, defined in gx_host.cu).
constexpr uint32_t kErrConsumerWait = 1u;   // a consumer warp gave up waiting for a staged k-block or d_u tile
constexpr uint32_t kErrProducerWait = 2u;   // the producer gave up waiting for a free stage / d_u buffer
constexpr uint32_t kErrDrainWait = 4u;      // the producer gave up waiting for its own copies after an abort
// Informational (the results are still exact): a stream-kernel CTA's wait for the previous CTA's partial sums ran out
// (kHandoffTimeoutNs), so it computed that tile's whole chain itself.
constexpr uint32_t kErrHandoffRecomputed = 8u;
constexpr uint32_t kErrFatalMask = kErrConsumerWait | kErrProducerWait | kErrDrainWait;
constexpr int64_t kHandoffTimeoutNs = 1000000;   // 1 ms: a healthy hand-off waits microseconds

// Parameters of the TMA-fed kernel. The tensor maps describe x [n][j][i], d_dv [n][j][c] and d_u [n][i][c] as 3-D
// float32 tensors (innermost first: i / c, then rows, then chunks). Chunk coordinate of step-local chunk p:
// n_base + p. The epilogue stores to du + n*du_sn + i*du_si + c directly.
struct TmaParams {
    CUtensorMap tm_x;
    CUtensorMap tm_dv;
    CUtensorMap tm_du;
    CUtensorMap tm_x4;      // slab kernel: x as {32 rows, j, row block, n}, box = four 32-row slabs
    CUtensorMap tm_du1;     // slab kernel: d_u box of one 32-row slab
    float *du;
    int64_t du_sn, du_si;
    int32_t n_base;
    int32_t P, C, hd;
    int32_t nib, ncb;       // row blocks (ceil(C / TI)) and column blocks (ceil(hd / TC)) per chunk
    int32_t ntiles;         // P * nib * ncb
    int32_t prefetch;       // 1: prefetch the first tile's d_dv boxes into L2 before the dependency wait
    int64_t timeout_ns;     // bound of every mbarrier wait
    uint32_t *err;          // the device error word (kErr* bits)
    int32_t stall_test;     // 1: the producer withholds the first stage's copies (failure-detection test hook)
    int32_t handoff_test;   // 1: stream kernel: publishers store but never flag their partial sums (test hook)
    int32_t stream_kappa;   // stream kernel: the split's charge per tile boundary in a CTA's range (stream_kappa())
    // offset configurations (kind 3): floats (0..3) by which the rows of x, d_dv and d_u start past the 16-byte
    // boundary their tensor maps were encoded from
    int32_t off_x, off_v, off_u;
    // Optional per-CTA timeline (nullptr: off; tile and stream kernels). Launch li = n_base / P < trace_launches writes,
    // for its CTA b of G, four global-timer stamps (ns) at trace[(li * G + b) * 4 + k]: k = 0 the CTA's start, 1 its
    // consumer warp 0 past the dependency wait, 2 that warp holding its first staged data, 3 that warp done with its
    // last output (results issued or partial sums staged).
    unsigned long long *trace;
    int32_t trace_launches;
    // stream kernel only (the plan's workspace): partial sums [grid][TI][TC] of each CTA's leading piece, one flag
    // per CTA, and one launch counter (the epoch) per CTA
    float *part;
    uint32_t *flags;
    uint32_t *ctl;
};

// Parameters of the generic kernel (any strides, 4-byte alignment).
struct GenericParams {
    float *du;
    const float *x;
    const float *dv;
    int64_t x_sn, x_sj, dv_sn, dv_sj, du_sn, du_si;
    int64_t x_si;           // element stride of x along i: 1, or the stored row stride when x is given transposed
    int64_t n_base;
    int32_t P, C, hd;
    int32_t nib, ncb;
    int32_t ntiles;
};

struct ConfigInfo {
    int TI, TC, KB, stages, threads, smem, RM, RN, consumer_warps;
    int eff;    // measured FMA-pipe efficiency (percent) with every SM busy
    int kind;   // 0: tile kernel; 1: balanced slab kernel (TI = slab rows; needs C % TI == 0 and C / TI >= 3);
                // 2: stream kernel (the step's (tile, j) work split evenly over the CTAs; needs a plan workspace);
                // 3: tile kernel for operand bases off a 16-byte boundary (aligned-down tensor maps)
    int shifted;   // kind 3: 0 element loads of boxes 4 floats wider; 1 tiles on the shifted grid
                   // (ceil((C + off_x) / TI) x ceil((hd + off_v) / TC) tiles a chunk; needs off_u == off_v)
    int tma_mid;   // 1 if the tiles a CTA finishes before its last (piece) are stored by TMA (kinds 0 and 2)
};

// Workspace of the stream kernel for `grid` CTAs of a TI x TC tile: partial sums [grid][TI][TC], one flag per CTA,
// one launch counter per CTA (each part 256-byte aligned).
inline size_t stream_workspace_bytes(int grid, int TI, int TC) {
    const size_t part = (static_cast<size_t>(grid) * TI * TC * 4 + 255) / 256 * 256;
    const size_t words = (static_cast<size_t>(grid) * 4 + 255) / 256 * 256;
    return part + 2 * words;
}

// The stream kernel's split of one step's work: W = ntiles x C units (tile t, j) in the order (t, j); CTA b of G takes
// units [b W / G, (b + 1) W / G). With W / G >= C its range is the tail of tile ta (j >= ja, continuing CTA b - 1's
// partial sums) if ja > 0, whole tiles, and the head of tile tb (j < je, whose partial sums CTA b + 1 continues) if
// je < C. Host and device share this code (the host exports it for tests).
struct Piece {
    int t;        // tile
    int j0, j1;   // j range [j0, j1)
    int kind;     // 0: whole tile; 1: head (publishes its partial sums); 2: tail (continues from CTA b - 1's)
};

struct Pieces {
    int ta, ja, tb, je;          // range [ta*C + ja, tb*C + je) of units (je in 1..C)
    int has_head, has_tail, first_full, nfull, count;
};

// unit u of the step at cost u + kappa * floor(u / C) (every tile begun after the first costs kappa units more) back
// from a cost y: inside tile t the cost runs t (C + kappa) .. t (C + kappa) + C; the kappa after it maps to the
// tile's end
template <class I>
__host__ __device__ inline I unit_at_cost(I y, I C, I kappa) {
    const I t = y / (C + kappa);
    const I r = y - t * (C + kappa);
    return t * C + (r < C ? r : C);
}

// CTA b takes the units between costs b F / G and (b + 1) F / G, F = the step's total cost: with kappa = 0 equal
// ranges of units; with kappa > 0 a range that holds a tile boundary (one more piece) holds kappa fewer units
template <class I>
__host__ __device__ inline Pieces cta_pieces_in(I ntiles, I C, I b, I G, I kappa) {
    const I F = ntiles * (C + kappa) - kappa;   // no charge after the last tile
    const I lo = unit_at_cost<I>(b * F / G, C, kappa);
    const I hi = unit_at_cost<I>((b + 1) * F / G, C, kappa);
    Pieces R;
    R.ta = static_cast<int>(lo / C);
    R.ja = static_cast<int>(lo - static_cast<I>(R.ta) * C);
    R.tb = static_cast<int>((hi - 1) / C);
    R.je = static_cast<int>(hi - static_cast<I>(R.tb) * C);
    R.has_tail = R.ja > 0 ? 1 : 0;
    R.has_head = R.je < C ? 1 : 0;
    R.first_full = R.has_tail ? R.ta + 1 : R.ta;
    const int last_full = R.has_head ? R.tb - 1 : R.tb;
    R.nfull = last_full >= R.first_full ? last_full - R.first_full + 1 : 0;
    R.count = R.has_head + R.nfull + R.has_tail;
    return R;
}

// In 32-bit arithmetic wherever G F fits: every thread of a stream-kernel CTA waits for this split before the first
// copy goes out, and on the large step the 64-bit divisions cost 0.25 us of each step (the CTAs that become resident
// last start on the critical path).
__host__ __device__ inline Pieces cta_pieces(int ntiles, int C, int b, int G, int kappa = 0) {
    const int64_t F = static_cast<int64_t>(ntiles) * (C + kappa) - kappa;
    if (F * G <= INT32_MAX) return cta_pieces_in<int32_t>(ntiles, C, b, G, kappa);
    return cta_pieces_in<int64_t>(ntiles, C, b, G, kappa);
}

// The split's charge per tile boundary (units of (tile, j)): a CTA whose range holds one more boundary runs one more
// piece (a publication or a reload of partial sums and an epilogue, ~1 us of stalled consumers on the large step), so
// it takes fewer units. Only when every range then stays longer than one tile (W / G >= C + 2 kappa).
#ifndef SDMGX_STREAM_KAPPA
#define SDMGX_STREAM_KAPPA 12
#endif
constexpr int kStreamKappa = SDMGX_STREAM_KAPPA;
inline int stream_kappa(int64_t ntiles, int C, int G) {
    return static_cast<int64_t>(ntiles) * C / G >= C + 2 * kStreamKappa ? kStreamKappa : 0;
}

// piece q of a CTA, in execution order: head, whole tiles, tail
__host__ __device__ inline Piece piece_at(const Pieces &R, int C, int q) {
    if (R.has_head) {
        if (q == 0) return Piece{R.tb, 0, R.je, 1};
        --q;
    }
    if (q < R.nfull) return Piece{R.first_full + q, 0, C, 0};
    return Piece{R.ta, R.ja, C, 2};
}

// TMA path
int tma_num_configs();
const ConfigInfo &tma_config(int k);
const void *tma_kernel(int k);
cudaError_t tma_launch(int k, const TmaParams &p, int grid, cudaStream_t st, int pdl);

// generic path (configs 0..2: 16, 32, 64 x 64 tiles; 3, the last: the 128 x 64 large-tile kernel)
int generic_num_configs();
const ConfigInfo &generic_config(int k);
const void *generic_kernel(int k);
cudaError_t generic_launch(int k, const GenericParams &p, int grid, cudaStream_t st, int pdl);

// synthetic successor (a consumer of d_u(ti) after the step)
cudaError_t successor_launch(const float *du, float *out, int64_t n0, int P, int hd, int64_t du_sn, cudaStream_t st,
                             int pdl, int sms);

// synthetic producer
cudaError_t producer_launch(float *dv, const float *S, int64_t base, int64_t count, int negate, cudaStream_t st,
                            int pdl, int sms);


}  // namespace sdmgx
