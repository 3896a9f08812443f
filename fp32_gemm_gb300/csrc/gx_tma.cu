// The TMA-fed, warp-specialised FP32 kernels of the gx_gemm step update (sm_103a): the tile kernel (gx_tma_kernel, with
// offset variants for operand bases off a 16-byte boundary, OCfg), the balanced slab kernel (gx_slab_kernel) and the
// stream kernel (gx_stream_kernel), which share the pipeline, the chain and the epilogue described here and differ in
// how a step's work is cut over the CTAs.
//
// What it computes (sparse_delta_memory/cuda/gx_gemm_cuda.py, module docstring formula and gx_gemm_kernel): for every
// chunk n of the step, row i < C and column c < hd, one thread runs acc = +0; acc = fmaf(x[n,j,i], d_dv[n,j,c], acc)
// for j = 0..C-1 in order, then writes d_u[n,i,c] + acc (one rounding). Tensor cores are not used: their rounding
// cannot reproduce that chain.
//
// How (our design for GB300, not the page's cp.async kernel):
//   * Persistent CTAs (grid <= resident slots) loop over tiles of TI rows x TC columns of one chunk.
//   * One producer warp (one elected lane) streams the operands with TMA (cp.async.bulk.tensor, 3-D tiled boxes of the
//     whole tensors, hardware zero fill past C / hd) into a ring of ST shared-memory stages of KB j-rows each:
//     xs[KB][TI] (x rows j, columns i) and ds[KB][TC] (d_dv rows j, columns c). mbarrier full/empty pairs with
//     transaction counts hand stages between producer and consumers. The d_u tile [TI][TC] is staged the same way.
//   * Consumer warps hold an RM x RN register tile per thread (4 x 8 lanes per warp, rows and columns in vectors of
//     up to 4) and run the j-chain in order with fmaf (rows in pairs as packed fma.rn.f32x2, bit-identical): per j,
//     RM/4 + RN/4 vector shared loads feed RM*RN FMAs.
//   * Programmatic dependent launch: before griddepcontrol.wait the producer issues the first tile's d_u box and the
//     x boxes of the first ST stages, and prefetches that tile's d_dv boxes into L2 (no visible effect: L2 is the
//     point of coherence). d_dv is loaded into shared memory only after the wait; d_u is written only after it.
//   * Every mbarrier wait is bounded (globaltimer); on expiry the thread sets a bit in the device error word and the
//     CTA unwinds; the producer first waits (bounded) for the copies it issued.
#include "gx_device.cuh"
#include "gx_internal.h"

namespace sdmgx {
namespace {

constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

template <int RM_, int RN_, int WM_, int WN_, int KB_, int ST_, int MINB_, int EFF_>
struct TCfg {
    static constexpr int EFF = EFF_;               // measured FMA-pipe efficiency at full occupancy, percent
    static constexpr int SLAB = 0;
    static constexpr bool ROWS_OUTER = false;      // FMA order within one j: column-outer (see chain_j)
    static constexpr bool TMID = false;            // tiles before a CTA's last stored by TMA (TmCfg, KCfg)
    static constexpr bool ELEM = false;            // offset configurations (OCfg): element loads of wide boxes
    static constexpr bool SHIFT = false;           // offset configurations (OCfg): tiles on the shifted grid
    static constexpr bool REALIGN = false;         // offset configurations (OCfg): wide boxes realigned per stage
    static constexpr bool UELEM = false;           // the staged d_u box is read, and d_u stored, element by element
    static constexpr int RM = RM_, RN = RN_;       // per-thread tile: rows x columns
    static constexpr int WM = WM_, WN = WN_;       // consumer warps along rows / columns
    static constexpr int KB = KB_, ST = ST_;       // j rows per stage, stages
    static constexpr int MINB = MINB_;             // CTAs per SM the register budget is sized for
    static constexpr int LM = 4, LN = 8;           // lanes along rows / columns
    static constexpr int VR = RM < 4 ? RM : 4, SR = RM / VR;
    static constexpr int VN = RN < 4 ? RN : 4, SN = RN / VN;
    static constexpr int TI = WM * RM * LM;
    static constexpr int TC = WN * RN * LN;
    static constexpr int NCW = WM * WN;
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int XP = TI, DP = TC, UP = TC;   // row pitches (floats) of the staged x, d_dv and d_u boxes
    // every TMA destination starts on a 128-byte boundary (the dynamic shared window is aligned up to 128 bytes)
    static constexpr int XS_BYTES = align_up(KB * TI * 4, 128);
    static constexpr int DS_BYTES = align_up(KB * TC * 4, 128);
    static constexpr int DU_BYTES = align_up(TI * TC * 4, 128);
    static constexpr int OFF_D = ST * XS_BYTES;
    static constexpr int OFF_U = OFF_D + ST * DS_BYTES;
    static constexpr int OFF_BAR = OFF_U + DU_BYTES;
    static constexpr int NBAR = 2 * ST + 2;
    static constexpr int SMEM = OFF_BAR + align_up(NBAR * 8, 128) + 128;   // + slack for the 128-byte alignment
    static constexpr uint32_t STAGE_TX = static_cast<uint32_t>(KB * (TI + TC) * 4);
    static constexpr uint32_t DU_TX = static_cast<uint32_t>(TI * TC * 4);
    static constexpr int UNROLL = (RM * RN >= 64) ? 8 : ((RM * RN >= 16) ? 16 : 32);
    static_assert(RM == 1 || RM == 2 || RM % 4 == 0, "RM: 1, 2 or a multiple of 4");
    static_assert(RN == 1 || RN == 2 || RN % 4 == 0, "RN: 1, 2 or a multiple of 4");
    static_assert(TI <= 256 && TC <= 256 && KB <= 256, "TMA box dimensions are at most 256");
    static_assert(TI % 4 == 0 && TC % 4 == 0, "box rows must be multiples of 16 bytes");
    static_assert(KB % UNROLL == 0 || UNROLL >= KB, "unroll divides KB");
};

struct Tile {
    int32_t n, i0, c0;
};

// One stamp of the optional timeline (see TmaParams::trace). Compiled only into the timeline build of the library
// (SDMGX_TRACE): even switched off at run time the stamps change the kernels' register allocation (2-3% on the large
// step, measured), so the default build has none. The CTA's index is re-read from the special registers.
#ifdef SDMGX_TRACE
constexpr bool kTrace = true;
#else
constexpr bool kTrace = false;
#endif
__device__ __forceinline__ void trace_at(const TmaParams &p, int k) {
    if constexpr (!kTrace) return;
    if (p.trace == nullptr) return;
    const int li = p.n_base / p.P;
    if (li < 0 || li >= p.trace_launches) return;
    const int G = static_cast<int>(gridDim.x);
    const int b = static_cast<int>(blockIdx.x);
    p.trace[(static_cast<int64_t>(li) * G + b) * 4 + k] = dev::global_timer_ns();
}

template <class Cfg>
__device__ __forceinline__ Tile decode_tile(const TmaParams &p, int t) {
    const int per_chunk = p.nib * p.ncb;
    const int pp = t / per_chunk;
    const int rem = t - pp * per_chunk;
    const int ib = rem / p.ncb;
    const int cb = rem - ib * p.ncb;
    return Tile{p.n_base + pp, ib * Cfg::TI, cb * Cfg::TC};
}

// V consecutive floats of a staged box: one vector load, or V element loads where the box rows sit one to three
// floats off a 16-byte boundary (the offset configurations).
template <class Cfg, int V>
__device__ __forceinline__ void lds(const float *p, float *o) {
    if constexpr (Cfg::ELEM) {
#pragma unroll
        for (int e = 0; e < V; ++e) o[e] = p[e];
    } else {
        dev::Vec<V>::load(p, o);
    }
}

// One j of the chain: the thread's x and d_dv fragments of row jj, then its RM x RN FMAs.
template <class Cfg>
__device__ __forceinline__ void chain_j(const float *__restrict__ xs, const float *__restrict__ ds, int jj,
                                        const int (&ro)[Cfg::SR], const int (&co)[Cfg::SN],
                                        float (&acc)[Cfg::RM][Cfg::RN]) {
    float a[Cfg::RM], b[Cfg::RN];
#pragma unroll
    for (int s = 0; s < Cfg::SR; ++s) lds<Cfg, Cfg::VR>(xs + jj * Cfg::XP + ro[s], a + s * Cfg::VR);
#pragma unroll
    for (int s = 0; s < Cfg::SN; ++s) lds<Cfg, Cfg::VN>(ds + jj * Cfg::DP + co[s], b + s * Cfg::VN);
    if constexpr (Cfg::RM % 2 == 0 && Cfg::ROWS_OUTER) {
        // rows in pairs, one row pair against all of the thread's columns before the next pair: the packed x pair
        // stays the same over RN consecutive FMAs (with 8 x 8 thread tiles the FMA pipe measured 89-90% busy inside
        // the pipeline, against 81-82% for the column-outer order of the 8 x 4 tiles)
#pragma unroll
        for (int r = 0; r < Cfg::RM; r += 2) {
#pragma unroll
            for (int c = 0; c < Cfg::RN; ++c) dev::fma2(acc[r][c], acc[r + 1][c], a[r], a[r + 1], b[c], b[c]);
        }
    } else if constexpr (Cfg::RM % 2 == 0) {
        // rows in pairs: (acc[r][c], acc[r+1][c]) += (a[r], a[r+1]) * (b[c], b[c]) with one packed FMA
#pragma unroll
        for (int c = 0; c < Cfg::RN; ++c) {
#pragma unroll
            for (int r = 0; r < Cfg::RM; r += 2) dev::fma2(acc[r][c], acc[r + 1][c], a[r], a[r + 1], b[c], b[c]);
        }
    } else {
#pragma unroll
        for (int r = 0; r < Cfg::RM; ++r) {
#pragma unroll
            for (int c = 0; c < Cfg::RN; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
        }
    }
}

// The chain for nj consecutive j of one stage (j order preserved: jj ascending).
//
// The same loop is spelt three ways because the compiler schedules them differently and each kernel family keeps
// the spelling it measured fastest with (differences of 1-2% on the large step, 17% on tiny steps):
//   * a full stage: the inline body under one unroll (tile and slab kernels), or the per-j helper (stream kernel, and
//     the tile kernel's rows-outer 8 x 8 configuration);
//   * a partial stage (the ragged end of C, or the end of a piece in the stream kernel): blocks of four unrolled j,
//     then one at a time (stream kernel and the small tiles, where C below the stage size makes every stage
//     partial), or the full-stage loop with a run-time count (the large tiles and the slab kernel, whose full stages
//     lose when the blocked form is compiled beside them).
template <class Cfg, bool FULL>
__device__ __forceinline__ void chain_block(const float *__restrict__ xs, const float *__restrict__ ds,
                                            const int (&ro)[Cfg::SR], const int (&co)[Cfg::SN],
                                            float (&acc)[Cfg::RM][Cfg::RN], int nj) {
    constexpr bool kHelper = Cfg::SLAB == 2 || Cfg::ROWS_OUTER;
    constexpr bool kBlocked = Cfg::SLAB == 2 || (Cfg::SLAB == 0 && Cfg::RM * Cfg::RN < 32);
    if constexpr (FULL && kHelper) {
#pragma unroll(Cfg::UNROLL)
        for (int jj = 0; jj < Cfg::KB; ++jj) chain_j<Cfg>(xs, ds, jj, ro, co, acc);
    } else if constexpr (!FULL && kBlocked) {
        int jj = 0;
        for (; jj + 4 <= nj; jj += 4) {
#pragma unroll
            for (int u = 0; u < 4; ++u) chain_j<Cfg>(xs, ds, jj + u, ro, co, acc);
        }
#pragma unroll 1
        for (; jj < nj; ++jj) chain_j<Cfg>(xs, ds, jj, ro, co, acc);
    } else {
        const int cnt = FULL ? Cfg::KB : nj;
#pragma unroll(Cfg::UNROLL)
        for (int jj = 0; jj < cnt; ++jj) {
            float a[Cfg::RM], b[Cfg::RN];
#pragma unroll
            for (int s = 0; s < Cfg::SR; ++s) lds<Cfg, Cfg::VR>(xs + jj * Cfg::XP + ro[s], a + s * Cfg::VR);
#pragma unroll
            for (int s = 0; s < Cfg::SN; ++s) lds<Cfg, Cfg::VN>(ds + jj * Cfg::DP + co[s], b + s * Cfg::VN);
            if constexpr (Cfg::RM % 2 == 0) {
                // rows in pairs: (acc[r][c], acc[r+1][c]) += (a[r], a[r+1]) * (b[c], b[c]) with one packed FMA
#pragma unroll
                for (int c = 0; c < Cfg::RN; ++c) {
#pragma unroll
                    for (int r = 0; r < Cfg::RM; r += 2)
                        dev::fma2(acc[r][c], acc[r + 1][c], a[r], a[r + 1], b[c], b[c]);
                }
            } else {
#pragma unroll
                for (int r = 0; r < Cfg::RM; ++r) {
#pragma unroll
                    for (int c = 0; c < Cfg::RN; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
                }
            }
        }
    }
}

// Epilogue: d_u + acc with one rounding each (the staged d_u tile us[TI][TC]), stored straight to global memory with
// vector stores; a vector that straddles hd, or one whose d_u address is off a 16-byte boundary (element-load offset
// configurations), is stored element by element; rows outside 0..C-1 and columns outside 0..hd-1 are skipped.
// Shifted-grid configurations: the tile's output rows and columns start off_x and off_v (= off_u) before its box
// coordinates; its d_u vectors then sit on 16-byte boundaries again.
template <class Cfg>
__device__ __forceinline__ void epilogue(const TmaParams &p, const Tile &tl, const float *us, const int (&ro)[Cfg::SR],
                                         const int (&co)[Cfg::SN], const float (&acc)[Cfg::RM][Cfg::RN]) {
    const int ir0 = Cfg::SHIFT ? tl.i0 - p.off_x : tl.i0;
    const int cr0 = Cfg::SHIFT ? tl.c0 - p.off_v : tl.c0;
    constexpr bool vec = !Cfg::UELEM;
#pragma unroll
    for (int sr = 0; sr < Cfg::SR; ++sr) {
#pragma unroll
        for (int er = 0; er < Cfg::VR; ++er) {
            const int rl = ro[sr] + er;
            const int i = ir0 + rl;
            if (i >= p.C || (Cfg::SHIFT && i < 0)) continue;
            float *grow = p.du + static_cast<int64_t>(tl.n) * p.du_sn + static_cast<int64_t>(i) * p.du_si;
#pragma unroll
            for (int sc = 0; sc < Cfg::SN; ++sc) {
                const int cl = co[sc];
                const int c = cr0 + cl;
                if (c >= p.hd || (Cfg::SHIFT && c + Cfg::VN <= 0)) continue;
                float u[Cfg::VN], o[Cfg::VN];
                if constexpr (vec) {
                    dev::Vec<Cfg::VN>::load(us + rl * Cfg::UP + cl, u);
                } else {
#pragma unroll
                    for (int e = 0; e < Cfg::VN; ++e) u[e] = us[rl * Cfg::UP + cl + e];
                }
#pragma unroll
                for (int e = 0; e < Cfg::VN; ++e) o[e] = __fadd_rn(u[e], acc[sr * Cfg::VR + er][sc * Cfg::VN + e]);
                if (vec && c >= 0 && c + Cfg::VN <= p.hd) {
                    dev::Vec<Cfg::VN>::store(grow + c, o);
                } else {
#pragma unroll
                    for (int e = 0; e < Cfg::VN; ++e)
                        if (c + e >= 0 && c + e < p.hd) grow[c + e] = o[e];
                }
            }
        }
    }
}

// The epilogue of a tile stored by TMA (TMID configurations): d_u + acc, one rounding each, written back over the
// staged d_u tile us[TI][TC] at the thread's own positions. Rows and columns outside the operands are written too (on
// zero-filled d_u); the TMA store leaves them out.
template <class Cfg>
__device__ __forceinline__ void epilogue_to_smem(float *us, const int (&ro)[Cfg::SR], const int (&co)[Cfg::SN],
                                                 const float (&acc)[Cfg::RM][Cfg::RN]) {
#pragma unroll
    for (int sr = 0; sr < Cfg::SR; ++sr) {
#pragma unroll
        for (int er = 0; er < Cfg::VR; ++er) {
#pragma unroll
            for (int sc = 0; sc < Cfg::SN; ++sc) {
                float *q = us + (ro[sr] + er) * Cfg::UP + co[sc];
                float u[Cfg::VN], o[Cfg::VN];
                dev::Vec<Cfg::VN>::load(q, u);
#pragma unroll
                for (int e = 0; e < Cfg::VN; ++e) o[e] = __fadd_rn(u[e], acc[sr * Cfg::VR + er][sc * Cfg::VN + e]);
                dev::Vec<Cfg::VN>::store(q, o);
            }
        }
    }
}

// Realigning offset configurations: warp w shifts rows w, w + NCW, .. of the stage's x box [KB][TI + 4] (then of its
// d_dv box [KB][TC + 4]) left by the operand's offset (0..3 floats) into the aligned buffers xa [KB][TI], da [KB][TC].
// A row is one warp-wide pass: lane l reads the box row's 16-byte vector l, takes the next one from lane l + 1 (lane
// 31 reads vector 32, the box's extra 4 floats), and writes aligned vector l from the two.
template <int OFF>
__device__ __forceinline__ float4 shift_left(float4 a, float4 b) {
    if constexpr (OFF == 0) return a;
    if constexpr (OFF == 1) return make_float4(a.y, a.z, a.w, b.x);
    if constexpr (OFF == 2) return make_float4(a.z, a.w, b.x, b.y);
    return make_float4(a.w, b.x, b.y, b.z);
}

template <int W>
__device__ __forceinline__ void realign_rows(const float *raw, float *al, int rows, int off, int warp, int nwarps,
                                             int lane) {
    static_assert(W == 128, "a box row is one warp-wide pass of 16-byte vectors");
    for (int r = warp; r < rows; r += nwarps) {
        const float4 *src = reinterpret_cast<const float4 *>(raw + r * (W + 4));
        const float4 a = src[lane];
        float4 b;
        b.x = __shfl_down_sync(0xffffffffu, a.x, 1);
        b.y = __shfl_down_sync(0xffffffffu, a.y, 1);
        b.z = __shfl_down_sync(0xffffffffu, a.z, 1);
        b.w = __shfl_down_sync(0xffffffffu, a.w, 1);
        if (lane == 31) b = src[32];
        float4 o;
        switch (off) {
            case 0: o = shift_left<0>(a, b); break;
            case 1: o = shift_left<1>(a, b); break;
            case 2: o = shift_left<2>(a, b); break;
            default: o = shift_left<3>(a, b); break;
        }
        reinterpret_cast<float4 *>(al + r * W)[lane] = o;
    }
}

template <class Cfg>
__device__ __forceinline__ void realign_stage(const float *xr, const float *dr, float *xa, float *da, int off_x,
                                              int off_v, int warp, int lane) {
    realign_rows<Cfg::TI>(xr, xa, Cfg::KB, off_x, warp, Cfg::NCW, lane);
    realign_rows<Cfg::TC>(dr, da, Cfg::KB, off_v, (warp + Cfg::KB) % Cfg::NCW, Cfg::NCW, lane);
}

// Realigning configurations: stage iteration k's staged boxes (raw stage k % ST) into aligned buffer k % 3; then the
// raw stage is released to the producer and buffer k % 3 marked with this warp's arrival. False: the staged boxes never
// came (the device error word is set).
template <class Cfg>
__device__ __forceinline__ bool realign_ahead(const TmaParams &p, unsigned char *base_g, uint32_t bar0,
                                              uint32_t du_empty, int k, int warp, int lane) {
    const int s = k % Cfg::ST;
    if (!__all_sync(0xffffffffu,
                    dev::mbar_wait(bar0 + 8u * s, static_cast<uint32_t>(k / Cfg::ST) & 1u, p.timeout_ns))) {
        if (lane == 0) atomicOr(p.err, kErrConsumerWait);
        return false;
    }
    const float *xr = reinterpret_cast<const float *>(base_g + s * Cfg::XS_BYTES);
    const float *dr = reinterpret_cast<const float *>(base_g + Cfg::OFF_D + s * Cfg::DS_BYTES);
    float *xa = reinterpret_cast<float *>(base_g + Cfg::OFF_A + (k % 3) * Cfg::A_BYTES);
    realign_stage<Cfg>(xr, dr, xa, xa + Cfg::KB * Cfg::TI, p.off_x, p.off_v, warp, lane);
    __syncwarp();
    if (lane == 0) {
        dev::mbar_arrive(bar0 + 8u * (Cfg::ST + s));
        dev::mbar_arrive(du_empty + 8u + 8u * static_cast<uint32_t>(k % 3));
    }
    return true;
}

// Coordinates of a tile's d_u box: the tile's own, or on the shifted grid off_x rows before its row coordinate (the
// tile's first output row; a negative row coordinate reads zeros). The column coordinate is the tile's own: the
// shifted grid requires off_u == off_v, so the box's columns are the tile's.
template <class Cfg>
__device__ __forceinline__ int du_x(const TmaParams &, const Tile &tl) { return tl.c0; }
template <class Cfg>
__device__ __forceinline__ int du_y(const TmaParams &p, const Tile &tl) { return Cfg::SHIFT ? tl.i0 - p.off_x : tl.i0; }

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MINB) gx_tma_kernel(const __grid_constant__ TmaParams p) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_s = dev::smem_addr(smem_raw);
    const uint32_t base_s = (raw_s + 127u) & ~127u;
    unsigned char *const base_g = smem_raw + (base_s - raw_s);
    const uint32_t bar0 = base_s + Cfg::OFF_BAR;
    const uint32_t du_full = bar0 + 8u * (2 * Cfg::ST);
    const uint32_t du_empty = du_full + 8u;
    const int warp = static_cast<int>(threadIdx.x) / 32;
    const int lane = static_cast<int>(threadIdx.x) % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::ST; ++s) {
            dev::mbar_init(bar0 + 8u * s, 1);                       // full[s]: the producer's expect_tx arrive
            dev::mbar_init(bar0 + 8u * (Cfg::ST + s), Cfg::NCW);    // empty[s]: one arrive per consumer warp
        }
        dev::mbar_init(du_full, 1);
        dev::mbar_init(du_empty, Cfg::NCW);
        if constexpr (Cfg::REALIGN) {   // realigned[b]: every consumer warp has realigned its rows into buffer b
            for (int bsel = 0; bsel < 3; ++bsel) dev::mbar_init(du_empty + 8u + 8u * bsel, Cfg::NCW);
        }
        dev::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) trace_at(p, 0);

    const int nk = (p.C + Cfg::KB - 1) / Cfg::KB;

    if (warp == Cfg::NCW) {
        // ------------------------------------------------ producer ------------------------------------------------
        if (lane != 0) return;
        int t = static_cast<int>(blockIdx.x);
        int it = 0;          // stage iterations issued (over all tiles)
        int du_issued = 0;   // d_u boxes issued
        int npre = 0;        // stages of the first tile whose x box went out before the dependency wait
        bool ok = true;
        Tile tl0{0, 0, 0};   // the first tile (decoded before the wait, so that its d_dv boxes go out right after it)
        if (t < p.ntiles) {
            dev::prefetch_tensormap(&p.tm_x);
            dev::prefetch_tensormap(&p.tm_dv);
            dev::prefetch_tensormap(&p.tm_du);
            const Tile tl = decode_tile<Cfg>(p, t);
            tl0 = tl;
            // first what the first k-block needs (x now, d_dv into L2 for after the wait); the d_u box, needed only by
            // the epilogue, goes out last so that it does not delay the first stage
            npre = nk < Cfg::ST ? nk : Cfg::ST;
            for (int s = 0; s < npre; ++s) {
                dev::mbar_arrive_expect_tx(bar0 + 8u * s, Cfg::STAGE_TX);
                if (s == 0 && p.stall_test) continue;   // test hook: stage 0 never completes
                dev::tma_load_3d(base_s + s * Cfg::XS_BYTES, &p.tm_x, tl.i0, s * Cfg::KB, tl.n, bar0 + 8u * s);
            }
            if (p.prefetch) {
                for (int kb = 0; kb < nk; ++kb) dev::tma_prefetch_3d(&p.tm_dv, tl.c0, kb * Cfg::KB, tl.n);
            }
            dev::mbar_arrive_expect_tx(du_full, Cfg::DU_TX);
            dev::tma_load_3d(base_s + Cfg::OFF_U, &p.tm_du, du_x<Cfg>(p, tl), du_y<Cfg>(p, tl), tl.n, du_full);
            du_issued = 1;
        }
        dev::grid_dependency_wait();
        // the armed stages' d_dv boxes first: the first thing the consumers need after the wait
        for (int s = 0; s < npre; ++s) {
            if (s == 0 && p.stall_test) continue;
            dev::tma_load_3d(base_s + Cfg::OFF_D + s * Cfg::DS_BYTES, &p.tm_dv, tl0.c0, s * Cfg::KB, tl0.n,
                             bar0 + 8u * s);
        }
        dev::launch_dependents();
        for (int tk = 0; t < p.ntiles && ok; t += static_cast<int>(gridDim.x), ++tk) {
            const Tile tl = decode_tile<Cfg>(p, t);
            for (int kb = 0; kb < nk; ++kb, ++it) {
                const int s = it % Cfg::ST;
                const uint32_t ph = static_cast<uint32_t>(it / Cfg::ST) & 1u;
                const uint32_t full = bar0 + 8u * s;
                const uint32_t dst_d = base_s + Cfg::OFF_D + s * Cfg::DS_BYTES;
                if (it < npre) continue;   // armed before the wait, its d_dv box issued right after it
                if (!dev::mbar_wait(bar0 + 8u * (Cfg::ST + s), ph ^ 1u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                dev::mbar_arrive_expect_tx(full, Cfg::STAGE_TX);
                dev::tma_load_3d(base_s + s * Cfg::XS_BYTES, &p.tm_x, tl.i0, kb * Cfg::KB, tl.n, full);
                dev::tma_load_3d(dst_d, &p.tm_dv, tl.c0, kb * Cfg::KB, tl.n, full);
            }
            // The d_u box of this tile goes out after its k-blocks: the single d_u buffer is free once every consumer
            // warp has finished the previous tile's epilogue, and the consumers need it only after this tile's last
            // k-block. Issuing it here keeps the k-block stream running ahead across tile boundaries.
            if (ok && tk > 0) {
                if (!dev::mbar_wait(du_empty, static_cast<uint32_t>(tk - 1) & 1u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                if constexpr (Cfg::TMID) {
                    // the previous tile, written back over the d_u buffer by the consumers: one TMA store, read out of
                    // the buffer before this tile's d_u box goes into it
                    const Tile tp = decode_tile<Cfg>(p, t - static_cast<int>(gridDim.x));
                    dev::tma_store_3d(&p.tm_du, tp.c0, tp.i0, tp.n, base_s + Cfg::OFF_U);
                    dev::bulk_wait_read_all();
                }
                dev::mbar_arrive_expect_tx(du_full, Cfg::DU_TX);
                dev::tma_load_3d(base_s + Cfg::OFF_U, &p.tm_du, du_x<Cfg>(p, tl), du_y<Cfg>(p, tl), tl.n, du_full);
                ++du_issued;
            }
        }
        if (p.stall_test) ok = false;   // the test hook always unwinds: its consumers never took every stage
        if (!ok) {
            atomicOr(p.err, kErrProducerWait);
            // Unwind: wait for the copies this thread issued (the last use of every stage, the last d_u box), so that
            // no TMA write lands in shared memory after the CTA has exited. A failed wait can only happen at an
            // iteration >= npre, so every stage armed before the dependency wait has received its d_dv box too and
            // each drained phase does complete.
            const int lo = it - Cfg::ST > 0 ? it - Cfg::ST : 0;
            for (int k = lo; k < it; ++k) {
                if (!dev::mbar_wait(bar0 + 8u * (k % Cfg::ST), static_cast<uint32_t>(k / Cfg::ST) & 1u, p.timeout_ns))
                    atomicOr(p.err, kErrDrainWait);
            }
            if (du_issued > 0 && !dev::mbar_wait(du_full, static_cast<uint32_t>(du_issued - 1) & 1u, p.timeout_ns))
                atomicOr(p.err, kErrDrainWait);
        }
        if constexpr (Cfg::TMID) dev::bulk_wait_all();   // every store performed before the CTA ends
        return;
    }

    // -------------------------------------------------- consumers --------------------------------------------------
    const int wm = warp % Cfg::WM;
    const int wn = warp / Cfg::WM;
    const int lm = lane / Cfg::LN;
    const int ln = lane % Cfg::LN;
    int ro[Cfg::SR], co[Cfg::SN];
#pragma unroll
    for (int s = 0; s < Cfg::SR; ++s) ro[s] = wm * Cfg::RM * Cfg::LM + s * Cfg::VR * Cfg::LM + lm * Cfg::VR;
#pragma unroll
    for (int s = 0; s < Cfg::SN; ++s) co[s] = wn * Cfg::RN * Cfg::LN + s * Cfg::VN * Cfg::LN + ln * Cfg::VN;

    dev::grid_dependency_wait();   // d_u is written below only after the predecessor grid has completed
    if (threadIdx.x == 0) trace_at(p, 1);
    // element-load offset configurations: the wide boxes hold the tile from float off on (and the d_u box of the
    // realigning ones too)
    const int ox = Cfg::ELEM ? p.off_x : 0, ov = Cfg::ELEM ? p.off_v : 0;
    const float *const us = reinterpret_cast<const float *>(base_g + Cfg::OFF_U) + (Cfg::UELEM ? p.off_u : 0);
    // stage iterations of this CTA (realigning configurations look one ahead)
    const int it_total = static_cast<int>(blockIdx.x) < p.ntiles
                             ? ((p.ntiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1) * nk
                             : 0;
    int it = 0;
    int tk = 0;
    for (int t = static_cast<int>(blockIdx.x); t < p.ntiles; t += static_cast<int>(gridDim.x), ++tk) {
        const Tile tl = decode_tile<Cfg>(p, t);
        float acc[Cfg::RM][Cfg::RN];
#pragma unroll
        for (int r = 0; r < Cfg::RM; ++r) {
#pragma unroll
            for (int c = 0; c < Cfg::RN; ++c) acc[r][c] = 0.0f;   // +0: the chain's start value
        }
        for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = it % Cfg::ST;
            const uint32_t ph = static_cast<uint32_t>(it / Cfg::ST) & 1u;
            // warp-uniform decision: every lane leaves together or none does (realigning configurations wait for
            // the staged boxes when they realign them)
            if (!Cfg::REALIGN && !__all_sync(0xffffffffu, dev::mbar_wait(bar0 + 8u * s, ph, p.timeout_ns))) {
                if (lane == 0) atomicOr(p.err, kErrConsumerWait);
                return;
            }

            const float *xs = reinterpret_cast<const float *>(base_g + s * Cfg::XS_BYTES) + ox;
            const float *ds = reinterpret_cast<const float *>(base_g + Cfg::OFF_D + s * Cfg::DS_BYTES) + ov;
            if constexpr (Cfg::REALIGN) {
                // Realigned one stage ahead: stage it is computed from buffer it % 3, whose rows every warp wrote
                // during its previous iteration; once every warp's rows are there, this warp writes its rows of stage
                // it + 1 into buffer (it + 1) % 3. That buffer last held stage it - 2, and every warp finished
                // computing stage it - 2 before it realigned stage it (its arrival on buffer it % 3).
                if (it == 0 && !realign_ahead<Cfg>(p, base_g, bar0, du_empty, 0, warp, lane)) return;
                const uint32_t b = du_empty + 8u + 8u * static_cast<uint32_t>(it % 3);
                if (!__all_sync(0xffffffffu, dev::mbar_wait(b, static_cast<uint32_t>(it / 3) & 1u, p.timeout_ns))) {
                    if (lane == 0) atomicOr(p.err, kErrConsumerWait);
                    return;
                }
                if (it + 1 < it_total && !realign_ahead<Cfg>(p, base_g, bar0, du_empty, it + 1, warp, lane)) return;
                xs = reinterpret_cast<const float *>(base_g + Cfg::OFF_A + (it % 3) * Cfg::A_BYTES);
                ds = xs + Cfg::KB * Cfg::TI;
            }
            const int nj = p.C - kb * Cfg::KB;
            if (nj >= Cfg::KB) {
                chain_block<Cfg, true>(xs, ds, ro, co, acc, Cfg::KB);
            } else {
                chain_block<Cfg, false>(xs, ds, ro, co, acc, nj);
            }
            if constexpr (!Cfg::REALIGN) {
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(bar0 + 8u * (Cfg::ST + s));
            }
        }
        if (!__all_sync(0xffffffffu, dev::mbar_wait(du_full, static_cast<uint32_t>(tk) & 1u, p.timeout_ns))) {
            if (lane == 0) atomicOr(p.err, kErrConsumerWait);
            return;
        }
        if (Cfg::TMID && t + static_cast<int>(gridDim.x) < p.ntiles) {
            // a tile before the CTA's last: back over the d_u buffer, stored by the producer (TMID)
            epilogue_to_smem<Cfg>(const_cast<float *>(us), ro, co, acc);
            dev::fence_proxy_async_smem();
        } else {
            epilogue<Cfg>(p, tl, us, ro, co, acc);
        }
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(du_empty);
    }
    if (threadIdx.x == 0) trace_at(p, 3);
}



// ---- the slab kernel: the 128 x 128 tile kernel with its work balanced over the SMs -----------------------------------
// The step's work is cut into slabs of 32 rows x TC columns of one chunk, ordered (chunk, column block, row block), and
// CTA b takes slabs [b S / G, (b + 1) S / G): every SM gets the same work to within one slab, so no SM idles through a
// second round that others do not have. A CTA runs its range in rounds of four slabs; slab w of a round is computed by
// warps 4w .. 4w + 3, one per SM sub-partition, so a partial round still loads every sub-partition evenly. When a
// round's four slabs are consecutive row blocks of one (chunk, column block), it is staged exactly like a 128-row tile
// (one x box of four 32-row slabs, one d_dv box, one d_u box); otherwise per slab (x, d_u) and per distinct
// (chunk, column block) (d_dv, at most two per round: the host requires C / 32 >= 3).
template <int KB_, int ST_, int EFF_>
struct SCfg {
    static constexpr int SLAB = 1;
    static constexpr int EFF = EFF_;
    static constexpr bool ROWS_OUTER = false;
    static constexpr bool TMID = false;
    static constexpr int RM = 8, RN = 4, KB = KB_, ST = ST_;
    static constexpr int WS = 4, WN = 4;           // slabs per round, warps per slab
    static constexpr int LM = 4, LN = 8;
    static constexpr int VR = 4, SR = 2, VN = 4, SN = 1;
    static constexpr int TI = RM * LM;             // 32 rows per slab
    static constexpr int TC = WN * RN * LN;        // 128 columns
    static constexpr int NCW = WS * WN;            // 16 consumer warps
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr bool ELEM = false, SHIFT = false, REALIGN = false, UELEM = false;
    static constexpr int XP = TI, DP = TC, UP = TC;
    static constexpr int X_SLAB = KB * TI * 4;     // bytes of one slab's x rows per stage
    static constexpr int D_BOX = KB * TC * 4;
    static constexpr int U_SLAB = TI * TC * 4;
    static constexpr int XS_BYTES = WS * X_SLAB;
    static constexpr int DS_BYTES = 2 * D_BOX;     // at most two (chunk, column block) per round
    static constexpr int OFF_D = ST * XS_BYTES;
    static constexpr int OFF_U = OFF_D + ST * DS_BYTES;
    static constexpr int OFF_BAR = OFF_U + WS * U_SLAB;
    static constexpr int NBAR = 2 * ST + 2;
    static constexpr int SMEM = OFF_BAR + align_up(NBAR * 8, 128) + 128;
    static constexpr int UNROLL = 16;
};

struct RoundInfo {
    int first, cnt;
    bool full;         // four slabs, one (chunk, column block), consecutive row blocks
    int key0, nd;      // key of the first slab; distinct keys (1 or 2)
};

__device__ __forceinline__ RoundInfo round_info(const TmaParams &p, int s_begin, int s_end, int r) {
    RoundInfo R;
    R.first = s_begin + 4 * r;
    int cnt = s_end - R.first;
    R.cnt = cnt < 0 ? 0 : (cnt > 4 ? 4 : cnt);
    R.key0 = R.first / p.nib;
    R.nd = R.cnt > 0 && (R.first + R.cnt - 1) / p.nib != R.key0 ? 2 : 1;
    R.full = R.cnt == 4 && R.nd == 1;
    return R;
}

template <class Cfg>
__device__ __forceinline__ void slab_coords(const TmaParams &p, int s, int32_t *n, int32_t *i0, int32_t *c0) {
    const int key = s / p.nib;
    const int rb = s - key * p.nib;
    const int pp = key / p.ncb;
    const int cb = key - pp * p.ncb;
    *n = p.n_base + pp;
    *i0 = rb * Cfg::TI;
    *c0 = cb * Cfg::TC;
}

template <class Cfg>
__device__ __forceinline__ uint32_t slab_stage_tx(const RoundInfo &R) {
    return R.full ? static_cast<uint32_t>(Cfg::XS_BYTES + Cfg::D_BOX)
                  : static_cast<uint32_t>(R.cnt * Cfg::X_SLAB + R.nd * Cfg::D_BOX);
}

// x (and / or) d_dv boxes of k-block kb of round R into stage buffers xs / ds, completing on `full`
template <class Cfg>
__device__ __forceinline__ void slab_issue(const TmaParams &p, const RoundInfo &R, int kb, uint32_t xs, uint32_t ds,
                                           uint32_t full, bool with_x, bool with_d) {
    int32_t n, i0, c0;
    slab_coords<Cfg>(p, R.first, &n, &i0, &c0);
    if (with_x) {
        if (R.full) {
            dev::tma_load_4d(xs, &p.tm_x4, 0, kb * Cfg::KB, i0 / Cfg::TI, n, full);
        } else {
            for (int w = 0; w < R.cnt; ++w) {
                int32_t nw, iw, cw;
                slab_coords<Cfg>(p, R.first + w, &nw, &iw, &cw);
                dev::tma_load_3d(xs + w * Cfg::X_SLAB, &p.tm_x, iw, kb * Cfg::KB, nw, full);
            }
        }
    }
    if (with_d) {
        dev::tma_load_3d(ds, &p.tm_dv, c0, kb * Cfg::KB, n, full);
        if (R.nd == 2) {
            int32_t n1, i1, c1;
            slab_coords<Cfg>(p, R.first + R.cnt - 1, &n1, &i1, &c1);
            dev::tma_load_3d(ds + Cfg::D_BOX, &p.tm_dv, c1, kb * Cfg::KB, n1, full);
        }
    }
}

template <class Cfg>
__device__ __forceinline__ void slab_issue_du(const TmaParams &p, const RoundInfo &R, uint32_t us, uint32_t bar) {
    int32_t n, i0, c0;
    slab_coords<Cfg>(p, R.first, &n, &i0, &c0);
    if (R.full) {
        dev::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(Cfg::WS * Cfg::U_SLAB));
        dev::tma_load_3d(us, &p.tm_du, c0, i0, n, bar);
    } else {
        dev::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(R.cnt * Cfg::U_SLAB));
        for (int w = 0; w < R.cnt; ++w) {
            int32_t nw, iw, cw;
            slab_coords<Cfg>(p, R.first + w, &nw, &iw, &cw);
            dev::tma_load_3d(us + w * Cfg::U_SLAB, &p.tm_du1, cw, iw, nw, bar);
        }
    }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1) gx_slab_kernel(const __grid_constant__ TmaParams p) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_s = dev::smem_addr(smem_raw);
    const uint32_t base_s = (raw_s + 127u) & ~127u;
    unsigned char *const base_g = smem_raw + (base_s - raw_s);
    const uint32_t bar0 = base_s + Cfg::OFF_BAR;
    const uint32_t du_full = bar0 + 8u * (2 * Cfg::ST);
    const uint32_t du_empty = du_full + 8u;
    const int warp = static_cast<int>(threadIdx.x) / 32;
    const int lane = static_cast<int>(threadIdx.x) % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::ST; ++s) {
            dev::mbar_init(bar0 + 8u * s, 1);
            dev::mbar_init(bar0 + 8u * (Cfg::ST + s), Cfg::NCW);
        }
        dev::mbar_init(du_full, 1);
        dev::mbar_init(du_empty, Cfg::NCW);
        dev::fence_mbar_init();
    }
    __syncthreads();

    const int nk = (p.C + Cfg::KB - 1) / Cfg::KB;
    const int s_begin = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.ntiles / gridDim.x);
    const int s_end = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.ntiles / gridDim.x);
    const int nrounds = (s_end - s_begin + Cfg::WS - 1) / Cfg::WS;

    if (warp == Cfg::NCW) {
        // ------------------------------------------------ producer ------------------------------------------------
        if (lane != 0) return;
        const int total_it = nrounds * nk;
        const int npre = total_it < Cfg::ST ? total_it : Cfg::ST;
        int it = 0, du_issued = 0;
        bool ok = true;
        if (nrounds > 0) {
            dev::prefetch_tensormap(&p.tm_x);
            dev::prefetch_tensormap(&p.tm_x4);
            dev::prefetch_tensormap(&p.tm_dv);
            dev::prefetch_tensormap(&p.tm_du);
            dev::prefetch_tensormap(&p.tm_du1);
            for (int q = 0; q < npre; ++q) {
                const RoundInfo Rq = round_info(p, s_begin, s_end, q / nk);
                dev::mbar_arrive_expect_tx(bar0 + 8u * q, slab_stage_tx<Cfg>(Rq));
                if (q == 0 && p.stall_test) continue;   // test hook: stage 0 never completes
                slab_issue<Cfg>(p, Rq, q % nk, base_s + q * Cfg::XS_BYTES, 0u, bar0 + 8u * q, true, false);
            }
            const RoundInfo R0 = round_info(p, s_begin, s_end, 0);
            if (p.prefetch) {
                int32_t n, i0, c0;
                slab_coords<Cfg>(p, R0.first, &n, &i0, &c0);
                for (int kb = 0; kb < nk; ++kb) dev::tma_prefetch_3d(&p.tm_dv, c0, kb * Cfg::KB, n);
            }
            slab_issue_du<Cfg>(p, R0, base_s + Cfg::OFF_U, du_full);
            du_issued = 1;
        }
        dev::grid_dependency_wait();
        // the armed stages' d_dv boxes first: the first thing the consumers need after the wait
        for (int q = 0; q < npre; ++q) {
            if (q == 0 && p.stall_test) continue;
            slab_issue<Cfg>(p, round_info(p, s_begin, s_end, q / nk), q % nk, base_s + q * Cfg::XS_BYTES,
                            base_s + Cfg::OFF_D + q * Cfg::DS_BYTES, bar0 + 8u * q, false, true);
        }
        dev::launch_dependents();
        for (int r = 0; r < nrounds && ok; ++r) {
            const RoundInfo R = round_info(p, s_begin, s_end, r);
            for (int kb = 0; kb < nk; ++kb, ++it) {
                const int s = it % Cfg::ST;
                const uint32_t ph = static_cast<uint32_t>(it / Cfg::ST) & 1u;
                const uint32_t full = bar0 + 8u * s;
                const uint32_t xs = base_s + s * Cfg::XS_BYTES;
                const uint32_t ds = base_s + Cfg::OFF_D + s * Cfg::DS_BYTES;
                if (it < npre) continue;   // armed before the wait, its d_dv boxes issued right after it
                if (!dev::mbar_wait(bar0 + 8u * (Cfg::ST + s), ph ^ 1u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                dev::mbar_arrive_expect_tx(full, slab_stage_tx<Cfg>(R));
                slab_issue<Cfg>(p, R, kb, xs, ds, full, true, true);
            }
            if (ok && r > 0) {
                if (!dev::mbar_wait(du_empty, static_cast<uint32_t>(r - 1) & 1u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                slab_issue_du<Cfg>(p, R, base_s + Cfg::OFF_U, du_full);
                ++du_issued;
            }
        }
        if (p.stall_test) ok = false;   // the test hook always unwinds: its consumers never took every stage
        if (!ok) {
            atomicOr(p.err, kErrProducerWait);
            const int lo = it - Cfg::ST > 0 ? it - Cfg::ST : 0;
            for (int k = lo; k < it; ++k) {
                if (!dev::mbar_wait(bar0 + 8u * (k % Cfg::ST), static_cast<uint32_t>(k / Cfg::ST) & 1u, p.timeout_ns))
                    atomicOr(p.err, kErrDrainWait);
            }
            if (du_issued > 0 && !dev::mbar_wait(du_full, static_cast<uint32_t>(du_issued - 1) & 1u, p.timeout_ns))
                atomicOr(p.err, kErrDrainWait);
        }
        return;
    }

    // -------------------------------------------------- consumers --------------------------------------------------
    const int ws = warp / Cfg::WN;   // the slab of the round this warp computes
    const int wn = warp % Cfg::WN;   // its column group (== its sub-partition)
    const int lm = lane / Cfg::LN;
    const int ln = lane % Cfg::LN;
    int ro[Cfg::SR], co[Cfg::SN];
#pragma unroll
    for (int s = 0; s < Cfg::SR; ++s) ro[s] = s * Cfg::VR * Cfg::LM + lm * Cfg::VR;
    co[0] = wn * Cfg::RN * Cfg::LN + ln * Cfg::VN;

    dev::grid_dependency_wait();
    int it = 0;
    for (int r = 0; r < nrounds; ++r) {
        const RoundInfo R = round_info(p, s_begin, s_end, r);
        const bool active = ws < R.cnt;
        int32_t n, i0, c0;
        slab_coords<Cfg>(p, active ? R.first + ws : R.first, &n, &i0, &c0);
        const int dslot = (n - p.n_base) * p.ncb + c0 / Cfg::TC == R.key0 ? 0 : 1;
        float acc[Cfg::RM][Cfg::RN];
#pragma unroll
        for (int i = 0; i < Cfg::RM; ++i) {
#pragma unroll
            for (int c = 0; c < Cfg::RN; ++c) acc[i][c] = 0.0f;   // +0: the chain's start value
        }
        for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = it % Cfg::ST;
            const uint32_t ph = static_cast<uint32_t>(it / Cfg::ST) & 1u;
            if (!__all_sync(0xffffffffu, dev::mbar_wait(bar0 + 8u * s, ph, p.timeout_ns))) {
                if (lane == 0) atomicOr(p.err, kErrConsumerWait);
                return;
            }
            if (active) {
                const float *xs = reinterpret_cast<const float *>(base_g + s * Cfg::XS_BYTES + ws * Cfg::X_SLAB);
                const float *ds =
                    reinterpret_cast<const float *>(base_g + Cfg::OFF_D + s * Cfg::DS_BYTES + dslot * Cfg::D_BOX);
                const int nj = p.C - kb * Cfg::KB;
                if (nj >= Cfg::KB) {
                    chain_block<Cfg, true>(xs, ds, ro, co, acc, Cfg::KB);
                } else {
                    chain_block<Cfg, false>(xs, ds, ro, co, acc, nj);
                }
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(bar0 + 8u * (Cfg::ST + s));
        }
        if (!__all_sync(0xffffffffu, dev::mbar_wait(du_full, static_cast<uint32_t>(r) & 1u, p.timeout_ns))) {
            if (lane == 0) atomicOr(p.err, kErrConsumerWait);
            return;
        }
        if (active) {
            const Tile tl{n, i0, c0};
            const float *us = reinterpret_cast<const float *>(base_g + Cfg::OFF_U + ws * Cfg::U_SLAB);
            epilogue<Cfg>(p, tl, us, ro, co, acc);
        }
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(du_empty);
    }
}

// ---- the stream kernel: the tile kernel with the step's (tile, j) work split evenly over the CTAs ----------------------
// Every output's chain runs over j = 0..C-1 in order, but nothing requires one CTA to run all of it: a chain stopped
// after some j and continued later from the same FP32 accumulator value gives the same bits. So the step's work is laid
// out as W = tiles x C units (tile t, j) in the order (t, j), and CTA b takes a contiguous range of them, an equal
// share of the step's cost (the units plus a charge for each tile boundary inside a range, cta_pieces): the SMs get
// the same work to within that charge, where whole tiles leave 104 of 152 SMs with a second tile on the large shape.
// With W / G >= C (the host's condition) a CTA's range is, in order, the tail of a tile whose leading j belong to CTA
// b - 1, some whole tiles, and the leading j of a tile whose tail belongs to CTA b + 1 (cta_pieces). It runs them as
//   1. the head piece first: the first je values of j of its last tile, from +0. The consumer warps leave their
//      accumulators in the d_u buffer (idle until the first d_u box; fragment order, store_frag) and go on at once;
//      the publisher warp copies those TI x TC values to the workspace with one bulk store, waits for it, and marks
//      the CTA's flag with this launch's epoch; the producer issues the CTA's first d_u box only after that;
//   2. its whole tiles, as in the tile kernel;
//   3. the tail piece last: the producer waits (bounded) for CTA b - 1's flag, copies that CTA's partial sums into a
//      shared buffer of their own with one bulk copy, and the consumers continue the chain from them at j = ja, then
//      add d_u.
// TMID: a tile the CTA finishes before its last piece is not stored by the consumers: they write d_u + acc back over
// the staged d_u tile and go on at once, and the publisher warp stores it with one TMA store, handing the d_u buffer
// back to the producer once the store has read it. The CTA's last tile keeps the consumers' own stores, so that no
// store's completion lies between the CTA's last FMA and its end.
// CTA b - 1 finishes its head piece after ja units of work; CTA b starts its tail after (W / G) - (C - ja) >= ja units,
// so the hand-off is normally ready long before it is needed. Flags carry an epoch: each CTA counts the launches that
// used the workspace in its own control word, which its publisher warp reads and advances right after the
// grid-dependency wait (the next launch reads it only after this one has completed; every CTA of every launch counts,
// so all CTAs agree on the epoch). A flag left by an earlier launch, or by an aborted one, therefore never matches.
template <class T, int EFF_, bool RO_ = false, int UNROLL_ = T::UNROLL, bool TMID_ = false>
struct KCfg : T {
    static constexpr int SLAB = 2;
    static constexpr int EFF = EFF_;
    static constexpr bool ROWS_OUTER = RO_;
    static constexpr int UNROLL = UNROLL_;
    static constexpr bool TMID = TMID_;   // tiles finished before the CTA's last piece: stored by TMA (see above)
    static constexpr int THREADS = (T::NCW + 2) * 32;         // consumers, producer, publisher
    static constexpr int OFF_P = T::OFF_BAR;                  // the incoming partial sums [TI][TC]
    static constexpr int OFF_BAR = OFF_P + T::DU_BYTES;
    // stages full / empty, d_u full / empty, partial full, head staged, head stored, epoch known, tile staged
    static constexpr int NBAR = 2 * T::ST + 7;
    static constexpr int OFF_EPOCH = OFF_BAR + NBAR * 8;      // this launch's epoch, from the publisher to the producer
    static constexpr int OFF_RECOMP = OFF_EPOCH + 4;          // 1: the tail piece recomputes its tile (late hand-off)
    static constexpr int OFF_PIECES = align_up(OFF_RECOMP + 4, 16);   // the CTA's Pieces (computed once)
    static constexpr int SMEM = align_up(OFF_PIECES + static_cast<int>(sizeof(Pieces)), 128) + 128;
    static_assert((T::TI * T::TC * 4) % 16 == 0, "the partial-sum tile is copied in 16-byte units");
};

// A consumer thread's accumulators, kept in their own fragment order instead of the tile's row-major order: vector v
// (v = sr * RN + c) of thread tid holds rows sr*4 .. sr*4 + 3 of the thread's column c, and sits at float offset
// (v * NCW*32 + tid) * 4. Column runs of four rows match the register pairs of the packed FMA (rows r, r + 1), and a
// warp's 16-byte accesses to one v are 512 contiguous bytes (no bank conflicts). Both ends of a hand-off use the same
// thread mapping, so the partial sums never need the tile's own layout.
template <class Cfg>
__device__ __forceinline__ void store_frag(float *dst, int tid, const float (&acc)[Cfg::RM][Cfg::RN]) {
    static_assert(Cfg::RM % 4 == 0, "fragments are column runs of four rows");
#pragma unroll
    for (int sr = 0; sr < Cfg::RM / 4; ++sr) {
#pragma unroll
        for (int c = 0; c < Cfg::RN; ++c) {
            const float v4[4] = {acc[sr * 4][c], acc[sr * 4 + 1][c], acc[sr * 4 + 2][c], acc[sr * 4 + 3][c]};
            dev::Vec<4>::store(dst + ((sr * Cfg::RN + c) * Cfg::NCW * 32 + tid) * 4, v4);
        }
    }
}

template <class Cfg>
__device__ __forceinline__ void load_frag(const float *src, int tid, float (&acc)[Cfg::RM][Cfg::RN]) {
#pragma unroll
    for (int sr = 0; sr < Cfg::RM / 4; ++sr) {
#pragma unroll
        for (int c = 0; c < Cfg::RN; ++c) {
            float v4[4];
            dev::Vec<4>::load(src + ((sr * Cfg::RN + c) * Cfg::NCW * 32 + tid) * 4, v4);
            acc[sr * 4][c] = v4[0];
            acc[sr * 4 + 1][c] = v4[1];
            acc[sr * 4 + 2][c] = v4[2];
            acc[sr * 4 + 3][c] = v4[3];
        }
    }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MINB) gx_stream_kernel(const __grid_constant__ TmaParams p) {
    extern __shared__ unsigned char smem_raw[];
    const int vt = static_cast<int>(threadIdx.x);
    const uint32_t raw_s = dev::smem_addr(smem_raw);
    const uint32_t base_s = (raw_s + 127u) & ~127u;
    unsigned char *const base_g = smem_raw + (base_s - raw_s);
    const uint32_t bar0 = base_s + Cfg::OFF_BAR;
    const uint32_t du_full = bar0 + 8u * (2 * Cfg::ST);
    const uint32_t du_empty = du_full + 8u;
    const uint32_t part_full = du_empty + 8u;
    const uint32_t head_staged = part_full + 8u;   // NCW arrivals: the head's accumulators are in the d_u buffer
    const uint32_t head_stored = head_staged + 8u; // 1 arrival: the publisher's bulk store has read them
    const uint32_t epoch_known = head_stored + 8u; // 1 arrival: the publisher has put the epoch in shared memory
    const uint32_t tile_staged = epoch_known + 8u; // NCW arrivals: a tile for the publisher's TMA store (TMID)
    volatile uint32_t *const epoch_s = reinterpret_cast<volatile uint32_t *>(base_g + Cfg::OFF_EPOCH);
    volatile uint32_t *const recomp_s = reinterpret_cast<volatile uint32_t *>(base_g + Cfg::OFF_RECOMP);
    const int warp = vt / 32;
    const int lane = vt % 32;
    const int b = static_cast<int>(blockIdx.x);
    const int G = static_cast<int>(gridDim.x);

    if (vt == 0) {
        for (int s = 0; s < Cfg::ST; ++s) {
            dev::mbar_init(bar0 + 8u * s, 1);
            dev::mbar_init(bar0 + 8u * (Cfg::ST + s), Cfg::NCW);
        }
        dev::mbar_init(du_full, 1);
        // TMID: only the publisher frees the d_u buffer (after each TMA store has read it); the last tile's buffer is
        // never needed again
        dev::mbar_init(du_empty, Cfg::TMID ? 1 : Cfg::NCW);
        dev::mbar_init(part_full, 1);
        dev::mbar_init(head_staged, Cfg::NCW);
        dev::mbar_init(head_stored, 1);
        dev::mbar_init(epoch_known, 1);
        dev::mbar_init(tile_staged, Cfg::NCW);
        dev::fence_mbar_init();
    }
    // the CTA's range, decoded by another warp while thread 0 sets up the barriers (both sit before the first copy)
    if (vt == 32) *reinterpret_cast<Pieces *>(base_g + Cfg::OFF_PIECES) = cta_pieces(p.ntiles, p.C, b, G, p.stream_kappa);
    __syncthreads();
    if (vt == 0) trace_at(p, 0);
    // read from shared memory where needed, so that no thread keeps the descriptor in registers
    const Pieces &R = *reinterpret_cast<const Pieces *>(base_g + Cfg::OFF_PIECES);

    if (warp == Cfg::NCW + 1) {
        // ------------------------------------------------ publisher -----------------------------------------------
        if (lane != 0) return;
        dev::grid_dependency_wait();
        // this launch's epoch: the CTA's count of earlier launches, advanced at once (nothing else reads the word)
        const uint32_t epoch = *reinterpret_cast<volatile const uint32_t *>(p.ctl + b);
        *reinterpret_cast<volatile uint32_t *>(p.ctl + b) = epoch + 1u;
        *epoch_s = epoch;
        dev::mbar_arrive(epoch_known);
        if (R.has_head) {
            if (dev::mbar_wait(head_staged, 0u, p.timeout_ns)) {
                dev::bulk_store(p.part + static_cast<int64_t>(b) * Cfg::TI * Cfg::TC, base_s + Cfg::OFF_U,
                                Cfg::DU_TX);
                dev::bulk_wait_all();
                dev::fence_proxy_async_global();
                if (!p.handoff_test) dev::st_release_gpu(p.flags + b, epoch + 1u);
            } else {
                atomicOr(p.err, kErrConsumerWait);
            }
            dev::mbar_arrive(head_stored);   // the d_u buffer is free again (also after a failed wait: no copy ran)
        }
        if constexpr (Cfg::TMID) {
            // the tiles the CTA finishes before its last piece (every piece after the head but the last)
            int k = 0;
            for (int q = R.has_head; q < R.count - 1; ++q, ++k) {
                const Tile tl = decode_tile<Cfg>(p, piece_at(R, p.C, q).t);
                if (!dev::mbar_wait(tile_staged, static_cast<uint32_t>(k) & 1u, p.timeout_ns)) {
                    atomicOr(p.err, kErrConsumerWait);
                    break;
                }
                dev::tma_store_3d(&p.tm_du, tl.c0, tl.i0, tl.n, base_s + Cfg::OFF_U);
                dev::bulk_wait_read_all();
                dev::mbar_arrive(du_empty);
            }
            dev::bulk_wait_all();   // every store performed before the CTA ends
        }
        return;
    }

    if (warp == Cfg::NCW) {
        // ------------------------------------------------ producer ------------------------------------------------
        if (lane != 0) return;
        int it = 0;            // stage iterations issued (over all pieces)
        int du_issued = 0;     // d_u boxes issued
        int npre = 0;          // stages of piece 0 whose x box went out before the dependency wait
        bool du0_early = false;
        bool part_issued = false;
        bool ok = true;
        const Piece P0 = piece_at(R, p.C, 0);
        const Tile tl0 = decode_tile<Cfg>(p, P0.t);   // decoded before the wait: its d_dv boxes go out right after it
        {
            dev::prefetch_tensormap(&p.tm_x);
            dev::prefetch_tensormap(&p.tm_dv);
            dev::prefetch_tensormap(&p.tm_du);
            const Tile &tl = tl0;
            const int nkb0 = (P0.j1 - P0.j0 + Cfg::KB - 1) / Cfg::KB;
            npre = nkb0 < Cfg::ST ? nkb0 : Cfg::ST;
            for (int s = 0; s < npre; ++s) {
                dev::mbar_arrive_expect_tx(bar0 + 8u * s, Cfg::STAGE_TX);
                if (s == 0 && p.stall_test) continue;   // test hook: stage 0 never completes
                dev::tma_load_3d(base_s + s * Cfg::XS_BYTES, &p.tm_x, tl.i0, P0.j0 + s * Cfg::KB, tl.n, bar0 + 8u * s);
            }
            if (p.prefetch) {
                for (int kb = 0; kb < nkb0; ++kb) dev::tma_prefetch_3d(&p.tm_dv, tl.c0, P0.j0 + kb * Cfg::KB, tl.n);
            }
            if (P0.kind == 0) {   // d_u of a whole first tile: read before the wait (the caller's PDL contract)
                dev::mbar_arrive_expect_tx(du_full, Cfg::DU_TX);
                dev::tma_load_3d(base_s + Cfg::OFF_U, &p.tm_du, tl.c0, tl.i0, tl.n, du_full);
                du_issued = 1;
                du0_early = true;
            }
        }
        dev::grid_dependency_wait();
        // the armed stages' d_dv boxes first: the first thing the consumers need after the wait
        for (int s = 0; s < npre; ++s) {
            if (s == 0 && p.stall_test) continue;
            dev::tma_load_3d(base_s + Cfg::OFF_D + s * Cfg::DS_BYTES, &p.tm_dv, tl0.c0, P0.j0 + s * Cfg::KB, tl0.n,
                             bar0 + 8u * s);
        }
        dev::launch_dependents();
        for (int q = 0; q < R.count && ok; ++q) {
            const Piece P = piece_at(R, p.C, q);
            const Tile tl = decode_tile<Cfg>(p, P.t);
            int j0 = P.j0;   // the piece's first j (0 for a tail that recomputes its tile)
            if (P.kind == 2) {
                // the partial sums of CTA b - 1 (its head piece: this tile's j < ja)
                if (!dev::mbar_wait(epoch_known, 0u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                if (dev::wait_flag(p.flags + (b - 1), *epoch_s + 1u,
                                   p.timeout_ns < kHandoffTimeoutNs ? p.timeout_ns : kHandoffTimeoutNs)) {
                    *recomp_s = 0u;
                    dev::fence_proxy_async_global();
                    dev::mbar_arrive_expect_tx(part_full, Cfg::DU_TX);
                    dev::bulk_load(base_s + Cfg::OFF_P, p.part + static_cast<int64_t>(b - 1) * Cfg::TI * Cfg::TC,
                                   Cfg::DU_TX, part_full);
                    part_issued = true;
                } else {
                    // CTA b - 1's partial sums are late (not resident, delayed, or withheld by the test hook): this
                    // CTA runs the tile's whole chain itself, from j = 0 and +0, and the bits are the same. x and
                    // d_dv are read-only, and CTA b - 1 never writes this tile's d_u. The consumers learn it from
                    // recomp_s, ordered by the barrier's release / acquire.
                    atomicOr(p.err, kErrHandoffRecomputed);
                    *recomp_s = 1u;
                    dev::mbar_arrive(part_full);
                    j0 = 0;
                }
            }
            const int nkb = (P.j1 - j0 + Cfg::KB - 1) / Cfg::KB;
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int s = it % Cfg::ST;
                const uint32_t ph = static_cast<uint32_t>(it / Cfg::ST) & 1u;
                const uint32_t full = bar0 + 8u * s;
                const uint32_t dst_d = base_s + Cfg::OFF_D + s * Cfg::DS_BYTES;
                const int j = j0 + kb * Cfg::KB;
                if (it < npre) continue;   // armed before the wait, its d_dv box issued right after it
                if (!dev::mbar_wait(bar0 + 8u * (Cfg::ST + s), ph ^ 1u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                dev::mbar_arrive_expect_tx(full, Cfg::STAGE_TX);
                dev::tma_load_3d(base_s + s * Cfg::XS_BYTES, &p.tm_x, tl.i0, j, tl.n, full);
                dev::tma_load_3d(dst_d, &p.tm_dv, tl.c0, j, tl.n, full);
            }
            if (!ok) break;
            // d_u of a piece that ends its tile, after the piece's k-blocks (as in the tile kernel). The first box
            // waits until the publisher has stored the head's partial sums out of the d_u buffer.
            if (P.kind != 1 && !(q == 0 && du0_early)) {
                const bool waited = du_issued > 0
                                        ? dev::mbar_wait(du_empty, static_cast<uint32_t>(du_issued - 1) & 1u,
                                                         p.timeout_ns)
                                        : (!R.has_head || dev::mbar_wait(head_stored, 0u, p.timeout_ns));
                if (!waited) {
                    ok = false;
                    break;
                }
                dev::mbar_arrive_expect_tx(du_full, Cfg::DU_TX);
                dev::tma_load_3d(base_s + Cfg::OFF_U, &p.tm_du, tl.c0, tl.i0, tl.n, du_full);
                ++du_issued;
            }
        }
        if (p.stall_test) ok = false;   // the test hook always unwinds: its consumers never took every stage
        if (!ok) {
            atomicOr(p.err, kErrProducerWait);
            // Unwind as the tile kernel does: wait for the copies this thread issued before leaving.
            const int lo = it - Cfg::ST > 0 ? it - Cfg::ST : 0;
            for (int k = lo; k < it; ++k) {
                if (!dev::mbar_wait(bar0 + 8u * (k % Cfg::ST), static_cast<uint32_t>(k / Cfg::ST) & 1u, p.timeout_ns))
                    atomicOr(p.err, kErrDrainWait);
            }
            if (du_issued > 0 && !dev::mbar_wait(du_full, static_cast<uint32_t>(du_issued - 1) & 1u, p.timeout_ns))
                atomicOr(p.err, kErrDrainWait);
            if (part_issued && !dev::mbar_wait(part_full, 0u, p.timeout_ns)) atomicOr(p.err, kErrDrainWait);
        }
        return;
    }

    // -------------------------------------------------- consumers --------------------------------------------------
    const int wm = warp % Cfg::WM;
    const int wn = warp / Cfg::WM;
    const int lm = lane / Cfg::LN;
    const int ln = lane % Cfg::LN;
    int ro[Cfg::SR], co[Cfg::SN];
#pragma unroll
    for (int s = 0; s < Cfg::SR; ++s) ro[s] = wm * Cfg::RM * Cfg::LM + s * Cfg::VR * Cfg::LM + lm * Cfg::VR;
#pragma unroll
    for (int s = 0; s < Cfg::SN; ++s) co[s] = wn * Cfg::RN * Cfg::LN + s * Cfg::VN * Cfg::LN + ln * Cfg::VN;

    dev::grid_dependency_wait();   // the workspace and d_u are touched only after the predecessor grid has completed
    if (vt == 0) trace_at(p, 1);
    if (kTrace && warp == 0 && p.trace != nullptr) {
        // the timeline's first-data stamp: warp 0 waits for stage 0 here (its loop then passes at once)
        (void)__all_sync(0xffffffffu, dev::mbar_wait(bar0, 0u, p.timeout_ns));
        if (lane == 0) trace_at(p, 2);
    }
    float *const us = reinterpret_cast<float *>(base_g + Cfg::OFF_U);
    const float *const ps = reinterpret_cast<const float *>(base_g + Cfg::OFF_P);
    int it = 0;
    int du_used = 0;
    bool failed = false;
    for (int q = 0; q < R.count && !failed; ++q) {
        const Piece P = piece_at(R, p.C, q);
        const Tile tl = decode_tile<Cfg>(p, P.t);
        float acc[Cfg::RM][Cfg::RN];
        int j0 = P.j0;
        if (P.kind == 2) {
            if (!__all_sync(0xffffffffu, dev::mbar_wait(part_full, 0u, p.timeout_ns))) {
                failed = true;
                break;
            }
            if (__builtin_expect(*recomp_s != 0u, 0)) {   // the hand-off was late: the whole chain here, from +0
                j0 = 0;
#pragma unroll
                for (int r = 0; r < Cfg::RM; ++r) {
#pragma unroll
                    for (int c = 0; c < Cfg::RN; ++c) acc[r][c] = 0.0f;
                }
            } else {
                load_frag<Cfg>(ps, vt, acc);
            }
        } else {
#pragma unroll
            for (int r = 0; r < Cfg::RM; ++r) {
#pragma unroll
                for (int c = 0; c < Cfg::RN; ++c) acc[r][c] = 0.0f;   // +0: the chain's start value
            }
        }
        const int nkb = (P.j1 - j0 + Cfg::KB - 1) / Cfg::KB;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
            const int s = it % Cfg::ST;
            const uint32_t ph = static_cast<uint32_t>(it / Cfg::ST) & 1u;
            if (!__all_sync(0xffffffffu, dev::mbar_wait(bar0 + 8u * s, ph, p.timeout_ns))) {
                failed = true;
                break;
            }
            const float *xs = reinterpret_cast<const float *>(base_g + s * Cfg::XS_BYTES);
            const float *ds = reinterpret_cast<const float *>(base_g + Cfg::OFF_D + s * Cfg::DS_BYTES);
            const int nj = P.j1 - (j0 + kb * Cfg::KB);
            if (nj >= Cfg::KB) {
                chain_block<Cfg, true>(xs, ds, ro, co, acc, Cfg::KB);
            } else {
                chain_block<Cfg, false>(xs, ds, ro, co, acc, nj);
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(bar0 + 8u * (Cfg::ST + s));
        }
        if (failed) break;
        if (P.kind == 1) {
            // the head's accumulators into the (still idle) d_u buffer, visible to the publisher's bulk store
            store_frag<Cfg>(us, vt, acc);
            dev::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(head_staged);
            continue;
        }
        if (!__all_sync(0xffffffffu, dev::mbar_wait(du_full, static_cast<uint32_t>(du_used) & 1u, p.timeout_ns))) {
            failed = true;
            break;
        }
        if (Cfg::TMID && q < R.count - 1) {
            epilogue_to_smem<Cfg>(us, ro, co, acc);
            dev::fence_proxy_async_smem();   // the values are read by the publisher's TMA store
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(tile_staged);
        } else {
            epilogue<Cfg>(p, tl, us, ro, co, acc);
            __syncwarp();
            if (!Cfg::TMID && lane == 0) dev::mbar_arrive(du_empty);
        }
        ++du_used;
    }
    if (failed && lane == 0) atomicOr(p.err, kErrConsumerWait);
    if (vt == 0) trace_at(p, 3);
}

template <class Cfg>
cudaError_t launch_cfg(const TmaParams &p, int grid, cudaStream_t st, int pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if constexpr (Cfg::SLAB == 1) {
        return cudaLaunchKernelEx(&cfg, gx_slab_kernel<Cfg>, p);
    } else if constexpr (Cfg::SLAB == 2) {
        return cudaLaunchKernelEx(&cfg, gx_stream_kernel<Cfg>, p);
    } else {
        return cudaLaunchKernelEx(&cfg, gx_tma_kernel<Cfg>, p);
    }
}

template <class Cfg>
const void *kernel_of() {
    if constexpr (Cfg::SLAB == 1) {
        return reinterpret_cast<const void *>(&gx_slab_kernel<Cfg>);
    } else if constexpr (Cfg::SLAB == 2) {
        return reinterpret_cast<const void *>(&gx_stream_kernel<Cfg>);
    } else {
        return reinterpret_cast<const void *>(&gx_tma_kernel<Cfg>);
    }
}


template <class Cfg>
ConfigInfo info_of() {
    return ConfigInfo{Cfg::TI, Cfg::TC, Cfg::KB, Cfg::ST, Cfg::THREADS, Cfg::SMEM, Cfg::RM, Cfg::RN, Cfg::NCW,
                      Cfg::EFF, (Cfg::ELEM || Cfg::SHIFT || Cfg::REALIGN) ? 3 : Cfg::SLAB, Cfg::SHIFT ? 1 : 0,
                      Cfg::TMID ? 1 : 0};
}

// The tile menu: (RM, RN, WM, WN, KB, ST, MINB, EFF). EFF is a calibrated FMA-pipe efficiency (percent) used by the
// host's geometry rule: for the larger tiles it is what the configuration reached on a GB300 with every SM busy; for
// the small latency-oriented tiles it was fitted so that the rule reproduces the measured ordering of small steps.
using C0 = TCfg<8, 4, 4, 4, 16, 4, 1, 75>;   // 128 x 128, 16 consumer warps, 8 x 4 per thread
// Tile configurations that store the tiles a CTA finishes before its last by TMA: the consumers write d_u + acc back
// over the staged d_u box, and the producer stores it before it loads the next tile's d_u there. With 8 x 8 thread
// tiles they also run the stream kernel's form of the loop (rows-outer packed FMAs, the per-j helper, an unroll of 16).
// Measured on multi-round steps against the same tile without either (us a step):
//   128 x 128, 8 warps of 8 x 8: 23.2 against 24.8 on 256 x 128 x 128 (the 8 x 4 tile: 23.8), 61.8 against 67.4
//   (65.6) on 800 x 128 x 128, where the consumers' own stores of a tile take ~1 us;
//   128 x 64, 4 warps of 8 x 8: 22.8 on 256 x 128 x 128, the fastest tile there (plans without a workspace take it);
//   64 x 128, 4 warps of 8 x 8: 33.3 against 36.5 on 200 x 192 x 128, 62.2 against 69.7 on 200 x 192 x 256;
//   64 x 64 and 32 x 128, 4 warps of 4 x 8 (the stores only; the loop form made no difference): 1-5% faster on the
//   sweep's multi-round shapes (9.0 against 9.2 on 300 x 64 x 96, 30.7 against 32.0 on 600 x 96 x 128), 1% slower on
//   800 x 32 x 128. The 64 x 128 tile with 8 warps of 4 x 8 measured 2% slower with them and keeps its own stores.
template <class T, bool RO_, int UNROLL_ = T::UNROLL>
struct TmCfg : T {
    static constexpr bool ROWS_OUTER = RO_;
    static constexpr int UNROLL = UNROLL_;
    static constexpr bool TMID = true;
};
using C1 = TmCfg<TCfg<8, 8, 4, 2, 32, 3, 1, 73>, true, 16>;   // 128 x 128,  8 warps, 8 x 8 per thread
using C2 = TmCfg<TCfg<8, 8, 4, 1, 32, 3, 2, 70>, true, 16>;   // 128 x  64,  4 warps
using C3 = TmCfg<TCfg<8, 8, 2, 2, 32, 3, 2, 70>, true, 16>;   //  64 x 128,  4 warps
using C4 = TCfg<4, 8, 4, 2, 32, 3, 2, 70>;   //  64 x 128,  8 warps, 4 x 8 per thread
using C5 = TmCfg<TCfg<4, 8, 4, 1, 32, 4, 2, 66>, false>;       //  64 x  64,  4 warps
using C6 = TmCfg<TCfg<4, 8, 2, 2, 32, 4, 2, 66>, false>;       //  32 x 128,  4 warps
using C7 = TCfg<4, 4, 2, 2, 32, 2, 4, 60>;   //  32 x  64,  4 warps (latency-bound steps)
using C8 = TCfg<2, 4, 2, 2, 32, 2, 4, 28>;   //  16 x  64,  4 warps
using C9 = TCfg<4, 4, 1, 1, 32, 2, 8, 25>;   //  16 x  32,  1 warp
using C10 = TCfg<2, 4, 1, 1, 32, 2, 8, 20>;  //   8 x  32,  1 warp
using C11 = SCfg<32, 3, 72>;                  // balanced 32 x 128 slabs, 16 warps (rounds of four slabs)
using C12 = KCfg<C0, 72>;                     // C0's tile with the (tile, j) work split evenly over the CTAs
using C13 = KCfg<TCfg<8, 4, 4, 2, 16, 4, 2, 70>, 68>;   // the same split on 128 x 64 tiles, 8 warps, 2 CTAs per SM
// The split on 128 x 128 tiles with 8 consumer warps of 8 x 8 (rows-outer FMA order, KB = 32, 3 stages, 224 KB of
// shared memory, 127 registers): a third fewer shared loads per FMA than C12. Its tiles finished before a CTA's last
// piece go out by TMA store (TMID): with 8 warps the consumers' own stores of a tile took ~1.1 us (too few stores in
// flight), against ~0.6 us with C12's 16. Measured on the large step (256 tiles on 152 SMs): 21.7 us, against 21.8-21.9
// without the TMA stores and 22.2-22.3 for C12; reading half of each tile's d_u into registers during its last stage
// (161 registers) had made it 22.1 us.
using C14 = KCfg<TCfg<8, 8, 4, 2, 32, 3, 1, 80>, 70, true, 16, true>;

// The tile kernel for operands whose rows start 4, 8 or 12 bytes past a 16-byte boundary (a 4-byte-aligned base with
// strides that are multiples of 16 bytes: a slice at an odd offset, say). TMA needs 16-byte-aligned bases and innermost
// coordinates, so the host encodes each operand's map from its base rounded down to 16 bytes, with the innermost
// extent grown by the offset (off = 1..3 floats; the map's rows then overlap the previous row's last off floats, which
// are loaded and never used). Three ways to use such maps:
//   * element loads (MODE_ = 0): every box is 4 floats wider than the tile, so that a box at the tile's own
//     (aligned) coordinate holds the tile's columns from float off on; the consumers read the staged boxes at that
//     offset with element loads (vectors would straddle 16-byte boundaries) and store d_u element by element. The
//     tiles are the aligned kernel's; the chain's shared loads are four times as many.
//   * the shifted grid (MODE_ = 1): tiles are cut on the aligned-down maps' own grid, so tile (ib, cb) holds output
//     rows ib TI - off_x .. and columns cb TC - off_v .., x and d_dv boxes are the tile's own size and the chain is the
//     aligned kernel's, vector loads included; a step has ceil((C + off_x) / TI) x ceil((hd + off_v) / TC) tiles per
//     chunk (rows and columns outside the operands are computed on zeros and not stored). It needs off_u == off_v:
//     the d_u box is then the tile's own size at the tile's column coordinate, and the epilogue's vectors are aligned.
//     (A d_u box wider than the tile, covering any off_u, measured 12% slower on small steps whenever a box ran past
//     the operand's columns.)
//   * realigned stages (MODE_ = 2): the element-load layout's wide boxes, which the consumer warps shift onto 16-byte
//     boundaries one stage ahead into three aligned buffers (each warp a share of the rows, then an mbarrier that every
//     consumer warp arrives on), so that the chain runs the aligned kernel's vector loads; a tenth more shared-memory
//     traffic instead of four times the load instructions.
// With every offset 0 each is the tile kernel on a few idle columns.
template <class T, int EFF_, int MODE_>   // MODE_: 0 element loads, 1 shifted grid, 2 realigned stages
struct OCfg : T {
    static constexpr int EFF = EFF_;
    static constexpr bool ELEM = MODE_ == 0, SHIFT = MODE_ == 1, REALIGN = MODE_ == 2, UELEM = MODE_ != 1;
    static constexpr int RX = SHIFT ? T::TI : T::TI + 4, RD = SHIFT ? T::TC : T::TC + 4;   // staged box row pitches
    static constexpr int XP = ELEM ? RX : T::TI, DP = ELEM ? RD : T::TC;   // the pitches the chain reads with
    static constexpr int UP = SHIFT ? T::TC : T::TC + 4;
    static constexpr int XS_BYTES = align_up(T::KB * RX * 4, 128);
    static constexpr int DS_BYTES = align_up(T::KB * RD * 4, 128);
    static constexpr int DU_BYTES = align_up(T::TI * UP * 4, 128);
    static constexpr int A_BYTES = REALIGN ? T::KB * (T::TI + T::TC) * 4 : 0;   // one aligned buffer: x, then d_dv
    static constexpr int OFF_D = T::ST * XS_BYTES;
    static constexpr int OFF_U = OFF_D + T::ST * DS_BYTES;
    static constexpr int OFF_A = OFF_U + DU_BYTES;
    static constexpr int OFF_BAR = OFF_A + 3 * A_BYTES;
    static constexpr int NBAR = T::NBAR + (REALIGN ? 3 : 0);
    static constexpr int SMEM = OFF_BAR + align_up(NBAR * 8, 128) + 128;
    static constexpr uint32_t STAGE_TX = static_cast<uint32_t>(T::KB * (RX + RD) * 4);
    static constexpr uint32_t DU_TX = static_cast<uint32_t>(T::TI * UP * 4);
    static_assert(RX <= 256 && RD <= 256, "TMA box dimensions are at most 256");
    static_assert(!REALIGN || (T::TI == 128 && T::TC == 128 && T::KB % 4 == 0), "realigned rows: one warp pass each");
};
using C15 = OCfg<C0, 60, 2>;    // 128 x 128, 16 warps, realigned stages: steps that fill the SMs
using C16 = OCfg<C7, 50, 0>;    //  32 x  64, 4 warps, element loads
using C17 = OCfg<C7, 60, 1>;    //  32 x  64, 4 warps, shifted grid
using C18 = OCfg<C10, 20, 1>;   //   8 x  32, 1 warp, shifted grid: the smallest steps

struct Entry {
    ConfigInfo info;
    const void *fn;
    cudaError_t (*launch)(const TmaParams &, int, cudaStream_t, int);
};

#define SDMGX_ENTRY(C) Entry{info_of<C>(), kernel_of<C>(), &launch_cfg<C>}
const Entry kEntries[] = {SDMGX_ENTRY(C0), SDMGX_ENTRY(C1), SDMGX_ENTRY(C2), SDMGX_ENTRY(C3), SDMGX_ENTRY(C4),
                          SDMGX_ENTRY(C5), SDMGX_ENTRY(C6), SDMGX_ENTRY(C7), SDMGX_ENTRY(C8), SDMGX_ENTRY(C9),
                          SDMGX_ENTRY(C10), SDMGX_ENTRY(C11), SDMGX_ENTRY(C12), SDMGX_ENTRY(C13),
                          SDMGX_ENTRY(C14), SDMGX_ENTRY(C15), SDMGX_ENTRY(C16), SDMGX_ENTRY(C17),
                          SDMGX_ENTRY(C18)};
#undef SDMGX_ENTRY

}  // namespace

int tma_num_configs() { return static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0])); }
const ConfigInfo &tma_config(int k) { return kEntries[k].info; }
const void *tma_kernel(int k) { return kEntries[k].fn; }
cudaError_t tma_launch(int k, const TmaParams &p, int grid, cudaStream_t st, int pdl) {
    return kEntries[k].launch(p, grid, st, pdl);
}

}  // namespace sdmgx
