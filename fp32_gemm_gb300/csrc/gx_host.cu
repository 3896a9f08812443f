// Host side of the gx_gemm C ABI: argument validation, per-device state, tile-configuration choice (the plan
// cache's geometry rule), TMA descriptor encoding, plans and the multi-step driver.
//
// Follows the page's launcher and plan entry points (sparse_delta_memory/cuda/gx_gemm_cuda.py: gx_gemm's checks,
// set_smem, gx_gemm_plan / gx_gemm_plan_launch, make_step), re-designed as a C ABI: every argument check runs before
// any CUDA call and returns a status code instead of throwing; a plan is a host struct holding the validated
// pointers, the geometry and the encoded tensor maps, and a launch patches only the step's chunk offset.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "gx_internal.h"
#include "sdm_gx_gemm.h"

static_assert(sdmgx::kErrFatalMask == SDM_GX_ERR_FATAL_MASK &&
                  sdmgx::kErrHandoffRecomputed == SDM_GX_ERR_HANDOFF_RECOMPUTED,
              "the device error word's bits as the header documents them");

// The device error word: bits of sdmgx::kErr* set by kernels whose bounded waits expired. One word per device (each
// device's module instance has its own copy); its device address is looked up once per device.
__device__ uint32_t g_sdm_gx_error_word;

namespace {

using namespace sdmgx;

constexpr int64_t kTwo31 = int64_t(1) << 31;
constexpr int64_t kMaxSpanElems = int64_t(1) << 60;
constexpr int64_t kMaxStride = int64_t(1) << 40;
constexpr int kMaxDevices = 64;
constexpr int kMaxConfigs = 32;
constexpr int64_t kWaitTimeoutNs = 2000000000LL;   // 2 s: a healthy wait lasts microseconds
constexpr int64_t kStallTestTimeoutNs = 20000000LL; // 20 ms under SDM_GX_FLAG_TEST_STALL
constexpr uint64_t kPlanMagic = 0x31504d4547584753ull;   // "SGXGEMP1"

thread_local int t_last_cuda = 0;
thread_local bool t_capturing = false;   // launches recorded into a graph are counted when the graph is launched
std::atomic<int64_t> g_count_step{0}, g_count_producer{0}, g_count_pdl{0}, g_count_succ{0};

int fail_cuda(cudaError_t e) {
    t_last_cuda = static_cast<int>(e);
    return SDM_GX_E_CUDA;
}

struct DevState {
    bool init = false;
    int status = 0;
    int sms = 0, optin = 0, smem_per_sm = 0, major = 0, minor = 0;
    uint32_t *err = nullptr;
    bool slab_ok = false;   // the driver accepts the slab kernel's 4-D x view (checked once)
    int tma_occ[kMaxConfigs] = {};
    int gen_occ[kMaxConfigs] = {};
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// x viewed as {32 rows, j, row block, n} (innermost first): one box of {32, KB, 4, 1} lands as four slabs of
// [KB][32] one after the other in shared memory.
CUresult encode_x_slabs(CUtensorMap *m, const float *base, int64_t C, int64_t chunks, int64_t sj, int64_t sn, int KB) {
    cuuint64_t dims[4] = {32u, static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(C / 32),
                          static_cast<cuuint64_t>(chunks)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(sj) * 4u, 128u, static_cast<cuuint64_t>(sn) * 4u};
    cuuint32_t box[4] = {32u, static_cast<cuuint32_t>(KB), 4u, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Per-device setup, once (under the lock): attributes, the error word's address, every kernel's shared-memory
// attribute and occupancy. Returns a status; *out points at the device's state.
int device_state(int *dev_out, const DevState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return SDM_GX_E_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState &d = g_dev[dev];
    if (!d.init) {
        DevState n;
        if ((e = cudaDeviceGetAttribute(&n.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&n.optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&n.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&n.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&n.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return fail_cuda(e);
        if (n.major != 10 || n.minor != 3) {
            n.status = SDM_GX_E_UNSUPPORTED;
            n.init = true;
            d = n;
            *dev_out = dev;
            *out = &d;
            return d.status;
        }
        if ((e = cudaGetSymbolAddress(reinterpret_cast<void **>(&n.err), g_sdm_gx_error_word)) != cudaSuccess)
            return fail_cuda(e);
        for (int k = 0; k < tma_num_configs() && k < kMaxConfigs; ++k) {
            const ConfigInfo &ci = tma_config(k);
            if (ci.smem > n.optin) continue;
            if ((e = cudaFuncSetAttribute(tma_kernel(k), cudaFuncAttributeMaxDynamicSharedMemorySize, ci.smem)) !=
                cudaSuccess)
                return fail_cuda(e);
            if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n.tma_occ[k], tma_kernel(k), ci.threads,
                                                                   ci.smem)) != cudaSuccess)
                return fail_cuda(e);
        }
        for (int k = 0; k < generic_num_configs() && k < kMaxConfigs; ++k) {
            const ConfigInfo &ci = generic_config(k);
            if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n.gen_occ[k], generic_kernel(k), ci.threads,
                                                                   0)) != cudaSuccess)
                return fail_cuda(e);
        }
        if (g_encode == nullptr) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q{};
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
                return fail_cuda(e != cudaSuccess ? e : cudaErrorNotSupported);
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        {   // encoding checks arguments only (no memory access): try the slab kernel's 4-D view on a dummy address
            CUtensorMap probe;
            n.slab_ok = encode_x_slabs(&probe, reinterpret_cast<const float *>(uintptr_t(1) << 20), 128, 2, 128,
                                       128 * 128, 32) == CUDA_SUCCESS;
        }
        n.init = true;
        d = n;
    }
    *dev_out = dev;
    *out = &d;
    return d.status;
}

// ---- validation -------------------------------------------------------------------------------------------------
struct Shape {
    int64_t N;        // chunks the operands hold (for _step: (ti + 1) * P, the minimum)
    int64_t P, C, hd;
    sdm_gx_strides s;
};

bool layout_ok(int64_t rows, int64_t cols, int64_t sr, int64_t sn, int64_t N) {
    if (sr < cols || sr > kMaxStride) return false;
    if (sn < rows * sr || sn > kMaxSpanElems / N) return false;
    return true;
}

struct Span {
    uintptr_t lo, hi;
};
Span span_of(const float *p, int64_t n0, int64_t n1, int64_t sn, int64_t sr, int64_t rows, int64_t cols) {
    const uintptr_t b = reinterpret_cast<uintptr_t>(p);
    return Span{b + static_cast<uintptr_t>(n0 * sn) * 4u,
                b + static_cast<uintptr_t>((n1 - 1) * sn + (rows - 1) * sr + cols) * 4u};
}
bool overlaps(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

// Checks shared by every entry point (before any CUDA call). n0 .. n1 - 1: the chunks whose spans must not overlap.
int validate(const float *du, const float *x, const float *dv, const Shape &sh, int64_t n0, int64_t n1) {
    if (du == nullptr || x == nullptr || dv == nullptr) return SDM_GX_E_NULL;
    if (sh.C < 1 || sh.C > 256 || sh.hd < 1 || sh.hd >= (int64_t(1) << 20)) return SDM_GX_E_SHAPE;
    const sdm_gx_strides &s = sh.s;
    if (!layout_ok(sh.C, sh.C, s.x_sj, s.x_sn, sh.N) || !layout_ok(sh.C, sh.hd, s.dv_sj, s.dv_sn, sh.N) ||
        !layout_ok(sh.C, sh.hd, s.du_si, s.du_sn, sh.N))
        return SDM_GX_E_STRIDE;
    if ((reinterpret_cast<uintptr_t>(du) | reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(dv)) & 3u)
        return SDM_GX_E_ALIGN;
    const Span su = span_of(du, n0, n1, s.du_sn, s.du_si, sh.C, sh.hd);
    const Span sx = span_of(x, n0, n1, s.x_sn, s.x_sj, sh.C, sh.C);
    const Span sv = span_of(dv, n0, n1, s.dv_sn, s.dv_sj, sh.C, sh.hd);
    if (overlaps(su, sx) || overlaps(su, sv)) return SDM_GX_E_OVERLAP;
    return SDM_GX_OK;
}

sdm_gx_strides contiguous(int64_t C, int64_t hd) {
    sdm_gx_strides s;
    s.x_sn = C * C;
    s.x_sj = C;
    s.dv_sn = C * hd;
    s.dv_sj = hd;
    s.du_sn = C * hd;
    s.du_si = hd;
    return s;
}

// Strides a tensor map can describe: multiples of 16 bytes, below 2^40 bytes.
bool tma_strides_ok(const sdm_gx_strides &s) {
    const int64_t st = s.x_sn | s.x_sj | s.dv_sn | s.dv_sj | s.du_sn | s.du_si;
    if (st & 3) return false;
    const int64_t mx = std::max({s.x_sn, s.x_sj, s.dv_sn, s.dv_sj, s.du_sn, s.du_si});
    return mx * 4 < kMaxStride;
}

// The TMA kernels proper: every base on a 16-byte boundary.
bool tma_eligible(const float *du, const float *x, const float *dv, const sdm_gx_strides &s) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(du) | reinterpret_cast<uintptr_t>(x) |
                        reinterpret_cast<uintptr_t>(dv);
    return (a & 15u) == 0 && tma_strides_ok(s);
}

// The offset configurations: TMA strides, some base 4, 8 or 12 bytes past a 16-byte boundary (every base is 4-byte
// aligned after validate()).
bool tma_offset_eligible(const float *du, const float *x, const float *dv, const sdm_gx_strides &s) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(du) | reinterpret_cast<uintptr_t>(x) |
                        reinterpret_cast<uintptr_t>(dv);
    return (a & 15u) != 0 && tma_strides_ok(s);
}

// floats by which p lies past a 16-byte boundary (0..3)
int32_t floats_off(const void *p) { return static_cast<int32_t>((reinterpret_cast<uintptr_t>(p) & 15u) / 4u); }

// ---- the launch description ----------------------------------------------------------------------------------------
struct Launch {
    int path = 0, config = 0, grid = 0, device = 0;
    int64_t n_first = 0;   // chunk index of the tensor maps' / pointers' origin
    int32_t P = 0;
    TmaParams tma;
    GenericParams gen;
    sdm_gx_geom geom;
};

// The geometry rule (our re-derivation, for this kernel family, of the page's one-wave rows rule): estimate the step
// time of every configuration on this device and take the fastest. The model, in microseconds:
//   step = base + compute + exposed memory,
// compute = the busiest SM's FMA work at the configuration's rate plus a fixed cost per round of resident CTAs (tile
// kernels: pipeline fill, epilogue, the chain's dependent latency), per slab round, or per piece (stream kernel);
// exposed memory = the step's algorithmic bytes at 7 TB/s, of which a share shows in the step that shrinks with the
// rounds an SM runs (later rounds load while earlier ones compute).
// How a partial last wave lands (measured): leftover CTAs after the first full waves spread one per SM when they are
// fewer than half the SMs, and otherwise fill whole SMs (every slot of an SM whose CTAs finished together), so that
// the busiest SM runs a whole extra round. The constants were fitted by least squares (log error) to the measured step
// time of every configuration on 66 shapes (P 48 .. 800, C 32 .. 128, hd 64 .. 128), one GB300 at 2.05 GHz; held out
// by C, the fit picks within 2% of the fastest configuration on average.
namespace model {
constexpr double kClockMHz = 2050.0;
constexpr double kBaseUs = 1.217;            // launch gap and first data of a chained step
constexpr double kTileRoundCycles = 1230.0;  // per round of resident CTAs (tile kernels)
constexpr double kPieceCycles = 1990.0;      // per piece of the stream kernel's split (fill, hand-off, epilogue)
constexpr double kSlabRoundCycles = 2771.0;  // per round of four slabs
constexpr double kStreamFixedCycles = 7732.0;
constexpr double kMemExposed = 0.541;        // share of the step's bytes at kMemBytesPerUs left exposed by one round
constexpr double kMemBytesPerUs = 7.0e6;
// fitted FMA rate per SM, as a fraction of 128 lanes a cycle, by configuration (the order of the TMA configuration
// table); a configuration past the table falls back to its kernel's own efficiency figure. The two 128 x 128 stream
// configurations share the model's piece costs, so their rates alone rank them: 8 x 8 (14) above 8 x 4 (12), as
// measured wherever a stream configuration is the fastest (C >= 96: up to 7% faster; at C <= 64, where tile kernels
// win, between 6% faster and 11% slower); 14's rate is fitted to its own sweep times with the other constants fixed,
// and so is 1's (the 8 x 8 tile with its TMA stores, above the 8 x 4 tile's 0: faster on 84 of the sweep's 102 shapes)
constexpr double kRate[] = {0.797, 0.812, 0.829, 0.823, 0.763, 0.746, 0.731, 0.677, 0.433, 0.430, 0.365,
                            0.731, 1.000, 0.971, 1.045, 0.590, 0.480, 0.630, 0.305};
constexpr int kRates = static_cast<int>(sizeof(kRate) / sizeof(kRate[0]));
}  // namespace model

// Tiles on the busiest SM and the rounds it runs them in, for `tiles` CTAs of which an SM holds `occ` at once.
void busiest_sm(int64_t tiles, int occ, int sms, int64_t *per, int64_t *rounds, int64_t *resident) {
    const int64_t w = static_cast<int64_t>(sms) * occ;
    int64_t p;
    if (tiles <= w) {
        p = (tiles + sms - 1) / sms;
    } else {
        const int64_t full = tiles / w, left = tiles % w;
        p = full * occ;
        if (left) p += 2 * left > sms ? occ : (left + sms - 1) / sms;
    }
    const int64_t a = std::max<int64_t>(1, std::min<int64_t>(occ, p));
    *per = p;
    *rounds = (p + a - 1) / a;
    *resident = a;
}

double estimate_us(int k, const ConfigInfo &ci, int occ, int sms, int64_t P, int64_t C, int64_t hd) {
    const int64_t g = ci.kind == 3 && ci.shifted ? 3 : 0;   // the shifted grid's extra rows and columns, at most
    const int64_t tiles = P * ((C + g + ci.TI - 1) / ci.TI) * ((hd + g + ci.TC - 1) / ci.TC);
    const double tile_fma = static_cast<double>(ci.TI) * ci.TC * C;
    const double rate = 128.0 * (k < model::kRates ? model::kRate[k] : ci.eff / 100.0);
    double cycles;
    int64_t rounds;
    if (ci.kind == 1) {
        // balanced slabs: every SM gets at most ceil(slabs / SMs), in rounds of four on 16 warps; a partial round of
        // r slabs costs about 1 + 0.9 r slabs (its fixed part does not shrink with r)
        const int64_t per_sm = (tiles + sms - 1) / sms;
        const int64_t full = per_sm / 4, r = per_sm % 4;
        const double eq = 4.0 * static_cast<double>(full) + (r ? 1.0 + 0.9 * static_cast<double>(r) : 0.0);
        rounds = (per_sm + 3) / 4;
        cycles = eq * tile_fma / rate + static_cast<double>(rounds) * model::kSlabRoundCycles;
    } else if (ci.kind == 2) {
        // (tile, j) units split evenly over every resident CTA; each CTA runs its whole tiles and up to two partial
        // pieces
        const int per_sm = std::max(1, occ);
        const double units_sm = std::ceil(static_cast<double>(tiles) * static_cast<double>(C) / sms);
        rounds = static_cast<int64_t>(std::ceil(units_sm / per_sm / static_cast<double>(C))) + 1;
        cycles = units_sm * ci.TI * ci.TC / rate + static_cast<double>(rounds) * model::kPieceCycles +
                 model::kStreamFixedCycles;
    } else {
        // whole tiles; below four consumer warps resident an SM's FMA rate drops in proportion
        int64_t per, a;
        busiest_sm(tiles, occ, sms, &per, &rounds, &a);
        const double share = std::min(1.0, static_cast<double>(a * ci.consumer_warps) / 4.0);
        cycles = static_cast<double>(per) * tile_fma / (rate * share) +
                 static_cast<double>(rounds) * model::kTileRoundCycles;
    }
    const double bytes = static_cast<double>(P) * static_cast<double>(C * C + 3 * C * hd) * 4.0;
    return model::kBaseUs + cycles / model::kClockMHz +
           model::kMemExposed * bytes / model::kMemBytesPerUs / static_cast<double>(std::max<int64_t>(1, rounds));
}

// The slab kernel needs whole 32-row slabs (C % 32 == 0) and at most two (chunk, column block) per round of four
// consecutive slabs (C / 32 >= 3). The stream kernel runs `stream_ctas` CTAs (every resident slot: SMs x CTAs per
// SM), needs the plan's workspace sized for them (ws_bytes), and at least as many tiles as CTAs, so that every CTA's
// range of (tile, j) units is at least one tile long. A configuration whose consumers store every tile themselves is
// offered up to kStreamMaxTilesPerCta tiles a CTA: past that whole tiles leave at most a sixteenth of a round idle,
// less than the split's own cost per tile (measured with 8 x 4 tiles: 8192 chunks of 128 x 128 x 128, 54 tiles an SM,
// 584 us a step split against 568 on whole tiles). One that stores the tiles finished before a CTA's last piece by TMA
// has no such bound: with 8 x 8 tiles it measured 531 us there, and 139 / 200 / 269 us against 152 / 215 / 288 on
// whole tiles at 2048 / 3000 / 4096 chunks.
constexpr int64_t kStreamMaxTilesPerCta = 16;
bool config_eligible(const ConfigInfo &ci, int64_t P, int64_t C, int64_t hd, int stream_ctas, size_t ws_bytes) {
    if (ci.kind == 1) return C % ci.TI == 0 && C / ci.TI >= 3;
    if (ci.kind == 2) {
        const int64_t tiles = P * ((C + ci.TI - 1) / ci.TI) * ((hd + ci.TC - 1) / ci.TC);
        return stream_ctas >= 1 && tiles >= stream_ctas &&
               (ci.tma_mid || tiles <= kStreamMaxTilesPerCta * stream_ctas) &&
               ws_bytes >= stream_workspace_bytes(stream_ctas, ci.TI, ci.TC);
    }
    return true;
}

// the stream kernel's grid for configuration k on this device: one CTA per resident slot
int stream_ctas_of(const DevState &d, int k) { return d.sms * std::max(0, d.tma_occ[k]); }

// stream_ctas_only > 0: a stream configuration is admitted only if its split runs exactly that many CTAs (the shared
// static workspace of sdm_gx_gemm_step_noalloc, whose per-CTA launch counters stay equal only if every launch on it
// counts the same CTAs).
// offset: some operand base lies off a 16-byte boundary; only the offset configurations (kind 3) serve it, and only
// it takes them unless forced; shift_ok: d_u and d_dv lie equally far off (the shifted-grid ones need that).
int choose_tma_config(const DevState &d, int64_t P, int64_t C, int64_t hd, int forced, size_t ws_bytes,
                      int stream_ctas_only, bool offset = false, bool shift_ok = true) {
    if (forced >= 0) return forced;
    auto tiles_of = [&](const ConfigInfo &ci) {
        const int64_t g = ci.kind == 3 && ci.shifted ? 3 : 0;   // the shifted grid's extra rows and columns, at most
        return P * ((C + g + ci.TI - 1) / ci.TI) * ((hd + g + ci.TC - 1) / ci.TC);
    };
    auto usable = [&](int k) {
        const ConfigInfo &ci = tma_config(k);
        return d.tma_occ[k] >= 1 && (ci.kind == 3) == offset && (shift_ok || !(ci.kind == 3 && ci.shifted)) &&
               config_eligible(ci, P, C, hd, stream_ctas_of(d, k), ws_bytes) &&
               !(ci.kind == 2 && stream_ctas_only > 0 && stream_ctas_of(d, k) != stream_ctas_only) &&
               !(ci.kind == 1 && !d.slab_ok) && tiles_of(ci) < kTwo31;
    };
    // Small steps (no tile of 32+ outputs per thread fills the SMs): the step is bound by latency, and the measured
    // best is the tile configuration with the most tiles that still fit one wave (a tile per SM, or two one-warp
    // CTAs), i.e. the most parallel chains of the least work each. Among equally many tiles the smaller tile wins (a CTA's time follows
    // its tile's area, rows and columns past C and hd included: 128 x 64 tiles on C = 64 took 5.8 us a step where
    // 64 x 64 tiles took 4.2), then the more efficient configuration.
    // (A property of the step's shape, decided on the aligned tile kernels whatever the layout: the offset menu has no
    // tile of 32+ outputs per thread small enough to tell.)
    bool throughput = false;
    for (int k = 0; k < tma_num_configs(); ++k) {
        const ConfigInfo &ci = tma_config(k);
        if (ci.kind == 0 && d.tma_occ[k] >= 1 && ci.RM * ci.RN >= 32 && tiles_of(ci) >= d.sms) throughput = true;
    }
    if (!throughput) {
        int bk = -1;
        int64_t bt = 0;
        for (int k = 0; k < tma_num_configs(); ++k) {
            // the tile kernels only: the slab and stream kernels balance work over rounds of a full GPU (a slab
            // kernel picked here took 8.7 us a step at 16 x 192 x 128, where 64 x 64 tiles take 6.9)
            if (!usable(k) || tma_config(k).kind == 1 || tma_config(k).kind == 2) continue;
            const ConfigInfo &ci = tma_config(k);
            const int64_t t = tiles_of(ci);
            // one wave: a tile per SM, or two one-warp CTAs (64 threads; two share an SM at no cost: 64 x 32 x 16
            // on 256 tiles of 8 x 32 took 1.83 us a step, on 128 tiles of 16 x 32 2.07)
            if (t > (ci.consumer_warps == 1 ? 2 * static_cast<int64_t>(d.sms) : d.sms)) continue;
            const ConfigInfo &cb = tma_config(bk < 0 ? k : bk);
            const int area = ci.TI * ci.TC, barea = cb.TI * cb.TC;
            if (bk < 0 || t > bt || (t == bt && (area < barea || (area == barea && ci.eff > cb.eff)))) {
                bk = k;
                bt = t;
            }
        }
        // (offset layouts: the menu has no medium tile, so a wave less than half full of its few tiles goes to the
        // model instead: 48 x 64 x 128 would take one 128 x 128 tile a chunk, 9.5 us, against 4.4 for 32 x 64)
        if (bk >= 0 && !(offset && 2 * bt < d.sms)) return bk;
    }
    // Otherwise the step-time model's fastest configuration.
    double best = 1e300;
    int bk = -1;
    for (int k = 0; k < tma_num_configs(); ++k) {
        if (!usable(k)) continue;
        const double est = estimate_us(k, tma_config(k), d.tma_occ[k], d.sms, P, C, hd);
        if (est < best * 0.999) {
            best = est;
            bk = k;
        }
    }
    return bk;
}

int choose_generic_config(const DevState &d, int64_t P, int64_t C, int64_t hd, int forced, bool x_transposed = false) {
    if (forced >= 0) return forced;
    // a step whose 128 x 64 tiles fill the SMs runs the large-tile kernel (the last configuration); smaller steps the
    // smallest tile that still fits one wave of resident CTAs (latency-bound). x given transposed: the small-tile
    // kernels only (the large-tile kernel stages x rows with i fastest), the 64-row one for filling steps.
    const int big = generic_num_configs() - 1;
    const ConfigInfo &cg = generic_config(big);
    if (P * ((C + cg.TI - 1) / cg.TI) * ((hd + cg.TC - 1) / cg.TC) >= d.sms) return x_transposed ? big - 1 : big;
    for (int k = 0; k < big; ++k) {
        const ConfigInfo &ci = generic_config(k);
        const int64_t tiles = P * ((C + ci.TI - 1) / ci.TI) * ((hd + ci.TC - 1) / ci.TC);
        if (tiles <= static_cast<int64_t>(d.sms) * std::max(1, d.gen_occ[k])) return k;
    }
    return big - 1;
}

CUresult encode_map(CUtensorMap *m, const float *base, int64_t inner, int64_t rows, int64_t chunks, int64_t sr,
                    int64_t sn, int box_inner, int box_rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(chunks)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(sr) * 4u, static_cast<cuuint64_t>(sn) * 4u};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows), 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Build the launch description for chunks n_first .. n_first + n_count - 1 (pointers and tensor maps originate at
// n_first). Runs after validate(); makes CUDA calls (device state, descriptor encoding).
// ws / ws_bytes: the plan's workspace (or none). fixed_part_bytes != 0 puts the workspace's flags and launch counters
// at that fixed offset whatever the configuration, splitting the rest of the workspace between them (the shared static
// array of sdm_gx_gemm_step_noalloc), and stream_ctas_only (as for choose_tma_config) fixes the stream kernel's CTA
// count there.
int build_launch(float *du, const float *x, const float *dv, const Shape &sh, int64_t n_first, int64_t n_count,
                 unsigned flags, Launch *L, void *ws = nullptr, size_t ws_bytes = 0, size_t fixed_part_bytes = 0,
                 int stream_ctas_only = 0) {
    const unsigned known = SDM_GX_FLAG_GENERIC | SDM_GX_FLAG_NO_PREFETCH | SDM_GX_FLAG_CONFIG_MASK |
                           SDM_GX_FLAG_CTAS_MASK | SDM_GX_FLAG_TEST_STALL | SDM_GX_FLAG_X_TRANSPOSED |
                           SDM_GX_FLAG_TEST_NO_HANDOFF;
    if (flags & ~known) return SDM_GX_E_FLAGS;
    int dev = 0;
    const DevState *dsp = nullptr;
    int rc = device_state(&dev, &dsp);
    if (rc != SDM_GX_OK) return rc;
    const DevState &d = *dsp;
    // operands must be device memory of this device
    const void *ptrs[3] = {du, x, dv};
    for (const void *q : ptrs) {
        cudaPointerAttributes at{};
        cudaError_t e = cudaPointerGetAttributes(&at, q);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return SDM_GX_E_DEVICE;
        }
        if ((at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) || at.device != dev)
            return SDM_GX_E_DEVICE;
    }
    const sdm_gx_strides &s = sh.s;
    const int forced = static_cast<int>(flags & SDM_GX_FLAG_CONFIG_MASK) - 1;
    const int forced_occ = static_cast<int>((flags & SDM_GX_FLAG_CTAS_MASK) >> SDM_GX_FLAG_CTAS_SHIFT);
    const bool x_t = (flags & SDM_GX_FLAG_X_TRANSPOSED) != 0;   // x stored [n][i][j]: the generic kernels
    const bool tma_ok = !(flags & SDM_GX_FLAG_GENERIC) && !x_t;
    const bool offs = tma_ok && !tma_eligible(du, x, dv, s) && tma_offset_eligible(du, x, dv, s);
    const bool use_tma = tma_ok && (offs || tma_eligible(du, x, dv, s));
    Launch l;
    l.device = dev;
    l.n_first = n_first;
    l.P = static_cast<int32_t>(sh.P);
    float *du0 = du + n_first * s.du_sn;
    const float *x0 = x + n_first * s.x_sn;
    const float *dv0 = dv + n_first * s.dv_sn;
    const ConfigInfo *ci = nullptr;
    int occ = 0;
    if (use_tma) {
        if (forced >= tma_num_configs()) return SDM_GX_E_FLAGS;
        const bool shift_ok = floats_off(du0) == floats_off(dv0);
        const int k = choose_tma_config(d, sh.P, sh.C, sh.hd, forced, ws != nullptr ? ws_bytes : 0, stream_ctas_only,
                                        offs, shift_ok);
        if (k < 0) return SDM_GX_E_SMEM;
        ci = &tma_config(k);
        if ((offs && ci->kind != 3) || (ci->kind == 3 && ci->shifted && !shift_ok) ||
            !config_eligible(*ci, sh.P, sh.C, sh.hd, stream_ctas_of(d, k), ws != nullptr ? ws_bytes : 0) ||
            (ci->kind == 2 && stream_ctas_only > 0 && stream_ctas_of(d, k) != stream_ctas_only) ||
            (ci->kind == 1 && !d.slab_ok))
            return SDM_GX_E_FLAGS;
        if (ci->smem > d.optin || d.tma_occ[k] < 1) return SDM_GX_E_SMEM;
        occ = d.tma_occ[k];
        l.path = 1;
        l.config = k;
        TmaParams &t = l.tma;
        std::memset(&t, 0, sizeof(t));
        CUresult r;
        const int du_rows = ci->kind == 1 ? 4 * ci->TI : ci->TI;   // slab kernel: a full round is four slabs
        // offset configurations: each map from its base rounded down to 16 bytes, the innermost extent grown by the
        // offset; element-load ones take boxes 4 floats wider (the tile from float off of each box row on), shifted-
        // grid ones the tile's own boxes (off_u == off_v)
        const bool k3 = ci->kind == 3, shifted = k3 && ci->shifted;
        const int ox = k3 ? floats_off(x0) : 0, ov = k3 ? floats_off(dv0) : 0, ou = k3 ? floats_off(du0) : 0;
        const int wide = k3 && !shifted ? 4 : 0, wide_u = wide;
        t.off_x = ox;
        t.off_v = ov;
        t.off_u = ou;
        if ((r = encode_map(&t.tm_x, x0 - ox, sh.C + ox, sh.C, n_count, s.x_sj, s.x_sn, ci->TI + wide, ci->KB)) !=
                CUDA_SUCCESS ||
            (r = encode_map(&t.tm_dv, dv0 - ov, sh.hd + ov, sh.C, n_count, s.dv_sj, s.dv_sn, ci->TC + wide,
                            ci->KB)) != CUDA_SUCCESS ||
            (r = encode_map(&t.tm_du, du0 - ou, sh.hd + ou, sh.C, n_count, s.du_si, s.du_sn, ci->TC + wide_u,
                            du_rows)) != CUDA_SUCCESS ||
            (ci->kind == 1 &&
             ((r = encode_x_slabs(&t.tm_x4, x0, sh.C, n_count, s.x_sj, s.x_sn, ci->KB)) != CUDA_SUCCESS ||
              (r = encode_map(&t.tm_du1, du0, sh.hd, sh.C, n_count, s.du_si, s.du_sn, ci->TC, ci->TI)) !=
                  CUDA_SUCCESS)))
            return fail_cuda(r == CUDA_ERROR_INVALID_VALUE ? cudaErrorInvalidValue : cudaErrorUnknown);
        t.du = du0;
        t.du_sn = s.du_sn;
        t.du_si = s.du_si;
        t.P = static_cast<int32_t>(sh.P);
        t.C = static_cast<int32_t>(sh.C);
        t.hd = static_cast<int32_t>(sh.hd);
        t.nib = static_cast<int32_t>((sh.C + (shifted ? ox : 0) + ci->TI - 1) / ci->TI);
        t.ncb = static_cast<int32_t>((sh.hd + (shifted ? ov : 0) + ci->TC - 1) / ci->TC);
        const int64_t tiles = sh.P * t.nib * t.ncb;
        if (tiles >= kTwo31) return SDM_GX_E_GRID;
        t.ntiles = static_cast<int32_t>(tiles);
        t.prefetch = (flags & SDM_GX_FLAG_NO_PREFETCH) ? 0 : 1;
        t.timeout_ns = (flags & SDM_GX_FLAG_TEST_STALL) ? kStallTestTimeoutNs : kWaitTimeoutNs;
        t.err = d.err;
        t.stall_test = (flags & SDM_GX_FLAG_TEST_STALL) ? 1 : 0;
        t.handoff_test = (flags & SDM_GX_FLAG_TEST_NO_HANDOFF) ? 1 : 0;
        if (ci->kind == 2) {   // workspace: partial sums, flags, control words (sizes as stream_workspace_bytes)
            unsigned char *w = static_cast<unsigned char *>(ws);
            const int G = stream_ctas_of(d, k);
            const size_t need = (static_cast<size_t>(G) * ci->TI * ci->TC * 4 + 255) / 256 * 256;
            const size_t part = fixed_part_bytes ? fixed_part_bytes : need;
            const size_t fl = fixed_part_bytes ? (ws_bytes > part ? (ws_bytes - part) / 2 / 256 * 256 : 0)
                                               : (static_cast<size_t>(G) * 4 + 255) / 256 * 256;
            if (part < need || static_cast<size_t>(G) * 4 > fl || part + 2 * fl > ws_bytes) return SDM_GX_E_FLAGS;
            t.stream_kappa = stream_kappa(t.ntiles, t.C, G);
            t.part = reinterpret_cast<float *>(w);
            t.flags = reinterpret_cast<uint32_t *>(w + part);
            t.ctl = reinterpret_cast<uint32_t *>(w + part + fl);
        }
    } else {
        if (forced >= generic_num_configs() || (x_t && forced == generic_num_configs() - 1)) return SDM_GX_E_FLAGS;
        const int k = choose_generic_config(d, sh.P, sh.C, sh.hd, forced, x_t);
        ci = &generic_config(k);
        occ = std::max(1, d.gen_occ[k]);
        l.path = 0;
        l.config = k;
        GenericParams &g = l.gen;
        g.du = du0;
        g.x = x0;
        g.dv = dv0;
        g.x_sn = s.x_sn;
        g.x_sj = x_t ? 1 : s.x_sj;   // transposed: j is the stored rows' unit stride, x_sj their stride (along i)
        g.x_si = x_t ? s.x_sj : 1;
        g.dv_sn = s.dv_sn;
        g.dv_sj = s.dv_sj;
        g.du_sn = s.du_sn;
        g.du_si = s.du_si;
        g.P = static_cast<int32_t>(sh.P);
        g.C = static_cast<int32_t>(sh.C);
        g.hd = static_cast<int32_t>(sh.hd);
        g.nib = static_cast<int32_t>((sh.C + ci->TI - 1) / ci->TI);
        g.ncb = static_cast<int32_t>((sh.hd + ci->TC - 1) / ci->TC);
        const int64_t tiles = sh.P * g.nib * g.ncb;
        if (tiles >= kTwo31) return SDM_GX_E_GRID;
        g.ntiles = static_cast<int32_t>(tiles);
    }
    if (forced_occ > 0) occ = std::min(occ, forced_occ);
    const int64_t tiles = l.path ? l.tma.ntiles : l.gen.ntiles;
    const int64_t slots = static_cast<int64_t>(d.sms) * occ;
    // the stream kernel runs one CTA per resident slot (its workspace is sized for that grid's CTAs)
    l.grid = (ci->kind == 2 && l.path == 1) ? static_cast<int>(slots)
                                             : static_cast<int>(std::max<int64_t>(1, std::min(tiles, slots)));
    sdm_gx_geom &gm = l.geom;
    gm.path = l.path;
    gm.config = l.config;
    gm.TI = ci->TI;
    gm.TC = ci->TC;
    gm.KB = ci->KB;
    gm.stages = ci->stages;
    gm.threads = ci->threads;
    gm.smem_bytes = ci->smem;
    gm.tiles = tiles;
    gm.ctas = l.grid;
    gm.ctas_per_sm = occ;
    gm.sms = d.sms;
    gm.one_wave = tiles <= slots ? 1 : 0;
    *L = l;
    return SDM_GX_OK;
}

// dv_rewritten: the kernel right before this step writes the step's d_dv (the producer chain), so an L2 prefetch of
// d_dv before the dependency wait would fetch lines that are about to be replaced; it is skipped.
int launch(const Launch &l, int64_t ti, cudaStream_t st, int pdl, bool dv_rewritten = false) {
    const int64_t nb = ti * l.P - l.n_first;
    cudaError_t e;
    if (l.path == 1) {
        TmaParams p = l.tma;
        p.n_base = static_cast<int32_t>(nb);
        if (dv_rewritten) p.prefetch = 0;
        e = tma_launch(l.config, p, l.grid, st, pdl);
    } else {
        GenericParams p = l.gen;
        p.n_base = nb;
        e = generic_launch(l.config, p, l.grid, st, pdl);
    }
    if (e != cudaSuccess) return fail_cuda(e);
    if (!t_capturing) {
        g_count_step.fetch_add(1, std::memory_order_relaxed);
        if (pdl) g_count_pdl.fetch_add(1, std::memory_order_relaxed);
    }
    return SDM_GX_OK;
}

}  // namespace

// ======================================================= plans =======================================================
struct sdm_gx_plan {
    uint64_t magic;
    const sdm_gx_plan *self;
    int64_t N, P, C, hd, ti_max;
    Shape shape;
    float *du;
    const float *x;
    const float *dv;
    Launch launch;
};

namespace {
int plan_check(const sdm_gx_plan *pl) {
    if (pl == nullptr || pl->magic != kPlanMagic || pl->self != pl) return SDM_GX_E_PLAN;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev != pl->launch.device) return SDM_GX_E_PLAN_DEVICE;
    return SDM_GX_OK;
}
}  // namespace

extern "C" {

int sdm_gx_abi_version(void) { return SDM_GX_ABI_VERSION; }

int sdm_gx_gemm_step(float *d_u, const float *x, const float *d_dv, int64_t ti, int64_t P, int64_t C, int64_t hd,
                     cudaStream_t stream, int pdl) {
    if (d_u == nullptr || x == nullptr || d_dv == nullptr) return SDM_GX_E_NULL;
    if (C < 1 || C > 256 || hd < 1 || hd >= (int64_t(1) << 20)) return SDM_GX_E_SHAPE;
    if (P < 1 || P >= kTwo31 || ti < 0 || ti > (kTwo31 - 1) / P - 1) return SDM_GX_E_RANGE;
    Shape sh{(ti + 1) * P, P, C, hd, contiguous(C, hd)};
    int rc = validate(d_u, x, d_dv, sh, ti * P, (ti + 1) * P);
    if (rc != SDM_GX_OK) return rc;
    Launch l;
    rc = build_launch(d_u, x, d_dv, sh, ti * P, P, 0u, &l);
    if (rc != SDM_GX_OK) return rc;
    return launch(l, ti, stream, pdl);
}

static int ex_common(float *d_u, const float *x, const float *d_dv, int64_t ti, int64_t N, int64_t P, int64_t C,
                     int64_t hd, const sdm_gx_strides *strides, Shape *sh) {
    if (d_u == nullptr || x == nullptr || d_dv == nullptr) return SDM_GX_E_NULL;
    if (C < 1 || C > 256 || hd < 1 || hd >= (int64_t(1) << 20)) return SDM_GX_E_SHAPE;
    if (N < 1 || N >= kTwo31 || P < 1 || P > N || ti < 0 || ti >= N / P) return SDM_GX_E_RANGE;
    *sh = Shape{N, P, C, hd, strides ? *strides : contiguous(C, hd)};
    return validate(d_u, x, d_dv, *sh, 0, N);
}

int sdm_gx_gemm_step_ex(float *d_u, const float *x, const float *d_dv, int64_t ti, int64_t N, int64_t P, int64_t C,
                        int64_t hd, const sdm_gx_strides *strides, cudaStream_t stream, int pdl, unsigned flags) {
    Shape sh;
    int rc = ex_common(d_u, x, d_dv, ti, N, P, C, hd, strides, &sh);
    if (rc != SDM_GX_OK) return rc;
    Launch l;
    rc = build_launch(d_u, x, d_dv, sh, ti * P, P, flags, &l);
    if (rc != SDM_GX_OK) return rc;
    return launch(l, ti, stream, pdl);
}

int noalloc_geometry(float *d_u, const float *x, const float *d_dv, const Shape &sh, Launch *l);

int sdm_gx_gemm_geometry(const float *d_u, const float *x, const float *d_dv, int64_t N, int64_t P, int64_t C,
                         int64_t hd, const sdm_gx_strides *strides, unsigned flags, sdm_gx_geom *out) {
    if (out == nullptr) return SDM_GX_E_NULL;
    Shape sh;
    int rc = ex_common(const_cast<float *>(d_u), x, d_dv, 0, N, P, C, hd, strides, &sh);
    if (rc != SDM_GX_OK) return rc;
    Launch l;
    if (flags & SDM_GX_FLAG_NOALLOC) {
        if (flags != SDM_GX_FLAG_NOALLOC) return SDM_GX_E_FLAGS;
        const sdm_gx_strides c = contiguous(C, hd);
        if (std::memcmp(&c, &sh.s, sizeof(c)) != 0) return SDM_GX_E_STRIDE;
        rc = noalloc_geometry(const_cast<float *>(d_u), x, d_dv, sh, &l);
        if (rc != SDM_GX_OK) return rc;
        *out = l.geom;
        return SDM_GX_OK;
    }
    rc = build_launch(const_cast<float *>(d_u), x, d_dv, sh, 0, N, flags, &l);
    if (rc != SDM_GX_OK) return rc;
    *out = l.geom;
    return SDM_GX_OK;
}

int sdm_gx_gemm_plan_workspace_size(const float *d_u, const float *x, const float *d_dv, int64_t N, int64_t P,
                                    int64_t C, int64_t hd, const sdm_gx_strides *strides, unsigned flags,
                                    size_t *bytes) {
    if (bytes == nullptr) return SDM_GX_E_NULL;
    *bytes = 0;
    Shape sh;
    int rc = ex_common(const_cast<float *>(d_u), x, d_dv, 0, N, P, C, hd, strides, &sh);
    if (rc != SDM_GX_OK) return rc;
    int dev = 0;
    const DevState *dsp = nullptr;
    rc = device_state(&dev, &dsp);
    if (rc != SDM_GX_OK) return rc;
    if ((flags & (SDM_GX_FLAG_GENERIC | SDM_GX_FLAG_X_TRANSPOSED)) || !tma_eligible(d_u, x, d_dv, sh.s)) return SDM_GX_OK;
    size_t need = 0;
    for (int k = 0; k < tma_num_configs(); ++k) {
        const ConfigInfo &ci = tma_config(k);
        if (ci.kind != 2 || dsp->tma_occ[k] < 1) continue;
        const int G = stream_ctas_of(*dsp, k);
        const size_t b = stream_workspace_bytes(G, ci.TI, ci.TC);
        if (config_eligible(ci, P, C, hd, G, b)) need = std::max(need, b);
    }
    *bytes = need;
    return SDM_GX_OK;
}

int sdm_gx_gemm_plan_create_ws(sdm_gx_plan **out, float *d_u, const float *x, const float *d_dv, int64_t N,
                               int64_t P, int64_t C, int64_t hd, const sdm_gx_strides *strides, int64_t ti_max,
                               unsigned flags, void *workspace, size_t workspace_bytes) {
    if (out == nullptr) return SDM_GX_E_NULL;
    *out = nullptr;
    Shape sh;
    int rc = ex_common(d_u, x, d_dv, ti_max, N, P, C, hd, strides, &sh);
    if (rc != SDM_GX_OK) return rc;
    if (workspace != nullptr) {
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return SDM_GX_E_ALIGN;
        const uintptr_t w0 = reinterpret_cast<uintptr_t>(workspace);
        const Span sw{w0, w0 + workspace_bytes};
        if (overlaps(sw, span_of(d_u, 0, sh.N, sh.s.du_sn, sh.s.du_si, sh.C, sh.hd)) ||
            overlaps(sw, span_of(x, 0, sh.N, sh.s.x_sn, sh.s.x_sj, sh.C, sh.C)) ||
            overlaps(sw, span_of(d_dv, 0, sh.N, sh.s.dv_sn, sh.s.dv_sj, sh.C, sh.hd)))
            return SDM_GX_E_OVERLAP;
    }
    Launch l;
    rc = build_launch(d_u, x, d_dv, sh, 0, N, flags, &l, workspace, workspace != nullptr ? workspace_bytes : 0);
    if (rc != SDM_GX_OK) return rc;
    if (l.path == 1 && tma_config(l.config).kind == 2) {
        // the workspace must be device memory of this device; its flags and control words start at zero (the
        // partial sums need no initial value), and the plan's first launch must see that
        cudaPointerAttributes at{};
        cudaError_t e = cudaPointerGetAttributes(&at, workspace);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return SDM_GX_E_DEVICE;
        }
        if ((at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) || at.device != l.device)
            return SDM_GX_E_DEVICE;
        unsigned char *ctl0 = reinterpret_cast<unsigned char *>(l.tma.flags);
        const size_t nctl = 2 * static_cast<size_t>(reinterpret_cast<unsigned char *>(l.tma.ctl) - ctl0);
        // synchronise first too: the caller's allocator may have handed out memory whose previous user still has
        // work in flight on another stream
        if ((e = cudaDeviceSynchronize()) != cudaSuccess || (e = cudaMemset(ctl0, 0, nctl)) != cudaSuccess ||
            (e = cudaDeviceSynchronize()) != cudaSuccess)
            return fail_cuda(e);
    }
    sdm_gx_plan *pl = static_cast<sdm_gx_plan *>(std::malloc(sizeof(sdm_gx_plan)));
    if (pl == nullptr) return SDM_GX_E_ALLOC;
    std::memset(static_cast<void *>(pl), 0, sizeof(*pl));
    pl->magic = kPlanMagic;
    pl->self = pl;
    pl->N = N;
    pl->P = P;
    pl->C = C;
    pl->hd = hd;
    pl->ti_max = ti_max;
    pl->shape = sh;
    pl->du = d_u;
    pl->x = x;
    pl->dv = d_dv;
    pl->launch = l;
    *out = pl;
    return SDM_GX_OK;
}

int sdm_gx_gemm_plan_create(sdm_gx_plan **out, float *d_u, const float *x, const float *d_dv, int64_t N, int64_t P,
                            int64_t C, int64_t hd, const sdm_gx_strides *strides, int64_t ti_max, unsigned flags) {
    return sdm_gx_gemm_plan_create_ws(out, d_u, x, d_dv, N, P, C, hd, strides, ti_max, flags, nullptr, 0);
}

int sdm_gx_gemm_plan_step(const sdm_gx_plan *plan, int64_t ti, cudaStream_t stream, int pdl) {
    int rc = plan_check(plan);
    if (rc != SDM_GX_OK) return rc;
    if (ti < 0 || ti > plan->ti_max) return SDM_GX_E_PLAN_TI;
    return launch(plan->launch, ti, stream, pdl);
}

int sdm_gx_gemm_autotune(float *d_u, const float *x, const float *d_dv, int64_t N, int64_t P, int64_t C, int64_t hd,
                         const sdm_gx_strides *strides, unsigned flags, void *workspace, size_t workspace_bytes,
                         int steps, cudaStream_t stream, unsigned *flags_out, int32_t *config_out, float *us_out) {
    if (flags_out == nullptr) return SDM_GX_E_NULL;
    if (steps < 1 || steps > 4096) return SDM_GX_E_RANGE;
    if (flags & (SDM_GX_FLAG_CONFIG_MASK | SDM_GX_FLAG_TEST_STALL)) return SDM_GX_E_FLAGS;
    if (P < 1 || N < P) return SDM_GX_E_RANGE;
    const int64_t T = N / P;
    // the automatic plan validates every argument and names the path this shape and layout take
    sdm_gx_plan *pl = nullptr;
    int rc = sdm_gx_gemm_plan_create_ws(&pl, d_u, x, d_dv, N, P, C, hd, strides, T - 1, flags, workspace,
                                        workspace_bytes);
    if (rc != SDM_GX_OK) return rc;
    const int path = pl->launch.path;
    sdm_gx_gemm_plan_destroy(pl);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    if (e != cudaSuccess) {
        if (e0 != nullptr) cudaEventDestroy(e0);
        return fail_cuda(e);
    }
    int best = -1;
    float best_us = 0.0f;
    const int nk = sdm_gx_gemm_num_configs(path);
    for (int k = 0; k < nk && rc == SDM_GX_OK; ++k) {
        sdm_gx_plan *pk = nullptr;
        int r = sdm_gx_gemm_plan_create_ws(&pk, d_u, x, d_dv, N, P, C, hd, strides, T - 1,
                                           flags | static_cast<unsigned>(k + 1), workspace, workspace_bytes);
        if (r == SDM_GX_E_FLAGS || r == SDM_GX_E_SMEM) continue;   // not admitted here
        if (r != SDM_GX_OK) {
            rc = r;
            break;
        }
        float ms = 0.0f;
        for (int s = 0; s < 2 && r == SDM_GX_OK; ++s) r = sdm_gx_gemm_plan_step(pk, s % T, stream, 1);
        if (r == SDM_GX_OK && (e = cudaEventRecord(e0, stream)) != cudaSuccess) r = fail_cuda(e);
        for (int s = 0; s < steps && r == SDM_GX_OK; ++s) r = sdm_gx_gemm_plan_step(pk, s % T, stream, 1);
        if (r == SDM_GX_OK && (e = cudaEventRecord(e1, stream)) != cudaSuccess) r = fail_cuda(e);
        if (r == SDM_GX_OK && (e = cudaEventSynchronize(e1)) != cudaSuccess) r = fail_cuda(e);
        if (r == SDM_GX_OK && (e = cudaEventElapsedTime(&ms, e0, e1)) != cudaSuccess) r = fail_cuda(e);
        sdm_gx_gemm_plan_destroy(pk);   // host memory only: the launches hold copies of its parameters
        if (r != SDM_GX_OK) {
            rc = r;
            break;
        }
        const float us = ms * 1000.0f / static_cast<float>(steps);
        if (best < 0 || us < best_us) {
            best = k;
            best_us = us;
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (rc != SDM_GX_OK) return rc;
    uint32_t word = 0;
    if ((rc = sdm_gx_device_error(&word, 0)) != SDM_GX_OK) return rc;
    if (best < 0) return SDM_GX_E_SMEM;   // not reached: the automatic plan's configuration is among those timed
    *flags_out = flags | static_cast<unsigned>(best + 1);
    if (config_out != nullptr) *config_out = best;
    if (us_out != nullptr) *us_out = best_us;
    return SDM_GX_OK;
}

int sdm_gx_gemm_plan_run(const sdm_gx_plan *plan, int64_t ti_begin, int64_t ti_end, cudaStream_t stream, int pdl) {
    int rc = plan_check(plan);
    if (rc != SDM_GX_OK) return rc;
    const int64_t step = ti_begin <= ti_end ? 1 : -1;
    const int64_t lo = step > 0 ? ti_begin : ti_end + 1;
    const int64_t hi = step > 0 ? ti_end - 1 : ti_begin;
    if (ti_begin != ti_end && (lo < 0 || hi > plan->ti_max)) return SDM_GX_E_PLAN_TI;
    for (int64_t ti = ti_begin; ti != ti_end; ti += step) {
        rc = launch(plan->launch, ti, stream, pdl);
        if (rc != SDM_GX_OK) return rc;
    }
    return SDM_GX_OK;
}

int sdm_gx_gemm_plan_run_producer(const sdm_gx_plan *plan, const float *S, int64_t ti_begin, int64_t ti_end,
                                  cudaStream_t stream, int pdl) {
    int rc = plan_check(plan);
    if (rc != SDM_GX_OK) return rc;
    if (S == nullptr) return SDM_GX_E_NULL;
    if (reinterpret_cast<uintptr_t>(S) & 3u) return SDM_GX_E_ALIGN;
    const Shape &sh = plan->shape;
    if (sh.s.dv_sj != sh.hd || sh.s.dv_sn != sh.C * sh.hd) return SDM_GX_E_STRIDE;   // the producer is contiguous
    const Span ss = span_of(S, 0, sh.N, sh.s.dv_sn, sh.s.dv_sj, sh.C, sh.hd);
    const Span sv = span_of(plan->dv, 0, sh.N, sh.s.dv_sn, sh.s.dv_sj, sh.C, sh.hd);
    const Span su = span_of(plan->du, 0, sh.N, sh.s.du_sn, sh.s.du_si, sh.C, sh.hd);
    if (overlaps(ss, sv) || overlaps(ss, su)) return SDM_GX_E_OVERLAP;
    const int64_t step = ti_begin <= ti_end ? 1 : -1;
    const int64_t lo = step > 0 ? ti_begin : ti_end + 1;
    const int64_t hi = step > 0 ? ti_end - 1 : ti_begin;
    if (ti_begin != ti_end && (lo < 0 || hi > plan->ti_max)) return SDM_GX_E_PLAN_TI;
    const int64_t per_step = sh.P * sh.C * sh.hd;
    const int sms = g_dev[plan->launch.device].sms;
    for (int64_t ti = ti_begin; ti != ti_end; ti += step) {
        cudaError_t e = producer_launch(const_cast<float *>(plan->dv), S,
                                        ti * per_step, per_step, static_cast<int>(ti & 1), stream, pdl, sms);
        if (e != cudaSuccess) return fail_cuda(e);
        if (!t_capturing) {
            g_count_producer.fetch_add(1, std::memory_order_relaxed);
            if (pdl) g_count_pdl.fetch_add(1, std::memory_order_relaxed);
        }
        rc = launch(plan->launch, ti, stream, pdl, true);
        if (rc != SDM_GX_OK) return rc;
    }
    return SDM_GX_OK;
}

}  // extern "C"

struct sdm_gx_graph {
    uint64_t magic;
    const sdm_gx_graph *self;
    int device;
    cudaGraphExec_t exec;
    int64_t steps, producers, successors, pdl_launches;   // launches one replay makes
};

namespace {
constexpr uint64_t kGraphMagic = 0x3148504152475853ull;   // "SXGRAPH1"
}

extern "C" {

int sdm_gx_gemm_plan_graph_create(sdm_gx_graph **out, const sdm_gx_plan *plan, const float *S, float *succ_out,
                                  int64_t ti_begin, int64_t ti_end, int pdl) {
    if (out == nullptr) return SDM_GX_E_NULL;
    *out = nullptr;
    int rc = plan_check(plan);
    if (rc != SDM_GX_OK) return rc;
    const int64_t n = ti_begin <= ti_end ? ti_end - ti_begin : ti_begin - ti_end;
    cudaStream_t cs = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
    if (e != cudaSuccess) return fail_cuda(e);
    e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        cudaStreamDestroy(cs);
        return fail_cuda(e);
    }
    t_capturing = true;
    if (S != nullptr && succ_out != nullptr) {
        rc = SDM_GX_E_FLAGS;   // one synthetic neighbour per chain
    } else if (S != nullptr) {
        rc = sdm_gx_gemm_plan_run_producer(plan, S, ti_begin, ti_end, cs, pdl);
    } else if (succ_out != nullptr) {
        rc = sdm_gx_gemm_plan_run_successor(plan, succ_out, ti_begin, ti_end, cs, pdl);
    } else {
        rc = sdm_gx_gemm_plan_run(plan, ti_begin, ti_end, cs, pdl);
    }
    t_capturing = false;
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(cs, &g);
    cudaStreamDestroy(cs);
    if (rc != SDM_GX_OK || e != cudaSuccess) {
        if (g != nullptr) cudaGraphDestroy(g);
        return rc != SDM_GX_OK ? rc : fail_cuda(e);
    }
    cudaGraphExec_t ex = nullptr;
    e = cudaGraphInstantiate(&ex, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return fail_cuda(e);
    sdm_gx_graph *gr = static_cast<sdm_gx_graph *>(std::malloc(sizeof(sdm_gx_graph)));
    if (gr == nullptr) {
        cudaGraphExecDestroy(ex);
        return SDM_GX_E_ALLOC;
    }
    gr->magic = kGraphMagic;
    gr->self = gr;
    gr->device = plan->launch.device;
    gr->exec = ex;
    gr->steps = n;
    gr->producers = S != nullptr ? n : 0;
    gr->successors = succ_out != nullptr ? n : 0;
    gr->pdl_launches = pdl ? n + gr->producers + gr->successors : 0;
    *out = gr;
    return SDM_GX_OK;
}

int sdm_gx_graph_launch(const sdm_gx_graph *graph, cudaStream_t stream) {
    if (graph == nullptr || graph->magic != kGraphMagic || graph->self != graph) return SDM_GX_E_PLAN;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev != graph->device) return SDM_GX_E_PLAN_DEVICE;
    e = cudaGraphLaunch(graph->exec, stream);
    if (e != cudaSuccess) return fail_cuda(e);
    if (!t_capturing) {
        g_count_step.fetch_add(graph->steps, std::memory_order_relaxed);
        g_count_producer.fetch_add(graph->producers, std::memory_order_relaxed);
        g_count_succ.fetch_add(graph->successors, std::memory_order_relaxed);
        g_count_pdl.fetch_add(graph->pdl_launches, std::memory_order_relaxed);
    }
    return SDM_GX_OK;
}

void sdm_gx_graph_destroy(sdm_gx_graph *graph) {
    if (graph == nullptr || graph->magic != kGraphMagic || graph->self != graph) return;
    cudaGraphExecDestroy(graph->exec);
    graph->magic = 0;
    graph->self = nullptr;
    std::free(graph);
}

int sdm_gx_gemm_plan_run_successor(const sdm_gx_plan *plan, float *out, int64_t ti_begin, int64_t ti_end,
                                   cudaStream_t stream, int pdl) {
    int rc = plan_check(plan);
    if (rc != SDM_GX_OK) return rc;
    if (out == nullptr) return SDM_GX_E_NULL;
    if (reinterpret_cast<uintptr_t>(out) & 3u) return SDM_GX_E_ALIGN;
    const Shape &sh = plan->shape;
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(out);
    const Span so{o0, o0 + static_cast<uintptr_t>(sh.N) * 4u};
    if (overlaps(so, span_of(plan->du, 0, sh.N, sh.s.du_sn, sh.s.du_si, sh.C, sh.hd)) ||
        overlaps(so, span_of(plan->x, 0, sh.N, sh.s.x_sn, sh.s.x_sj, sh.C, sh.C)) ||
        overlaps(so, span_of(plan->dv, 0, sh.N, sh.s.dv_sn, sh.s.dv_sj, sh.C, sh.hd)))
        return SDM_GX_E_OVERLAP;
    const int64_t step = ti_begin <= ti_end ? 1 : -1;
    const int64_t lo = step > 0 ? ti_begin : ti_end + 1;
    const int64_t hi = step > 0 ? ti_end - 1 : ti_begin;
    if (ti_begin != ti_end && (lo < 0 || hi > plan->ti_max)) return SDM_GX_E_PLAN_TI;
    const int sms = g_dev[plan->launch.device].sms;
    for (int64_t ti = ti_begin; ti != ti_end; ti += step) {
        rc = launch(plan->launch, ti, stream, pdl);
        if (rc != SDM_GX_OK) return rc;
        cudaError_t e = successor_launch(plan->du, out, ti * sh.P, static_cast<int>(sh.P), static_cast<int>(sh.hd),
                                         sh.s.du_sn, stream, pdl, sms);
        if (e != cudaSuccess) return fail_cuda(e);
        if (!t_capturing) {
            g_count_succ.fetch_add(1, std::memory_order_relaxed);
            if (pdl) g_count_pdl.fetch_add(1, std::memory_order_relaxed);
        }
    }
    return SDM_GX_OK;
}

int sdm_gx_gemm_plan_run_host(const sdm_gx_plan *plan, float *d_u_host, const float *x_host, const float *d_dv_host,
                              int64_t ti_begin, int64_t ti_end, cudaStream_t compute, cudaStream_t h2d,
                              cudaStream_t d2h) {
    int rc = plan_check(plan);
    if (rc != SDM_GX_OK) return rc;
    if (d_u_host == nullptr || x_host == nullptr || d_dv_host == nullptr) return SDM_GX_E_NULL;
    if (compute == h2d || compute == d2h || h2d == d2h) return SDM_GX_E_FLAGS;
    const Shape &sh = plan->shape;
    const sdm_gx_strides c = contiguous(sh.C, sh.hd);
    if (std::memcmp(&c, &sh.s, sizeof(c)) != 0) return SDM_GX_E_STRIDE;
    const int64_t step = ti_begin <= ti_end ? 1 : -1;
    const int64_t lo = step > 0 ? ti_begin : ti_end + 1;
    const int64_t hi = step > 0 ? ti_end - 1 : ti_begin;
    if (ti_begin != ti_end && (lo < 0 || hi > plan->ti_max)) return SDM_GX_E_PLAN_TI;
    const size_t xs = static_cast<size_t>(sh.P * sh.C * sh.C) * 4u;    // bytes of one step's x chunks
    const size_t vs = static_cast<size_t>(sh.P * sh.C * sh.hd) * 4u;   // bytes of one step's d_dv / d_u chunks
    cudaError_t e = cudaSuccess;
    {   // this call's copies in start after the work already on `compute` and `d2h` (an earlier call's last steps and
        // copies out still use the device tensors)
        cudaEvent_t prev_c = nullptr, prev_o = nullptr;
        if ((e = cudaEventCreateWithFlags(&prev_c, cudaEventDisableTiming)) != cudaSuccess) return fail_cuda(e);
        if ((e = cudaEventCreateWithFlags(&prev_o, cudaEventDisableTiming)) != cudaSuccess) {
            cudaEventDestroy(prev_c);
            return fail_cuda(e);
        }
        if ((e = cudaEventRecord(prev_c, compute)) == cudaSuccess && (e = cudaEventRecord(prev_o, d2h)) == cudaSuccess &&
            (e = cudaStreamWaitEvent(h2d, prev_c, 0)) == cudaSuccess)
            e = cudaStreamWaitEvent(h2d, prev_o, 0);
        cudaEventDestroy(prev_c);
        cudaEventDestroy(prev_o);
        if (e != cudaSuccess) return fail_cuda(e);
    }
    // consecutive steps are contiguous in memory: copy them in groups of about 16 MB, so that small steps do not
    // pay a copy's fixed cost each
    const int64_t per_step = static_cast<int64_t>(xs + 2 * vs);
    const int64_t group = std::max<int64_t>(1, (int64_t(16) << 20) / per_step);
    int64_t ti = ti_begin;
    while (ti != ti_end && e == cudaSuccess && rc == SDM_GX_OK) {
        int64_t cnt = step > 0 ? std::min(group, ti_end - ti) : std::min(group, ti - ti_end);
        const int64_t first = step > 0 ? ti : ti - cnt + 1;   // lowest step of the group (its memory starts there)
        const size_t ox = static_cast<size_t>(first) * xs / 4u, ov = static_cast<size_t>(first) * vs / 4u;
        const size_t nx = static_cast<size_t>(cnt) * xs, nv = static_cast<size_t>(cnt) * vs;
        cudaEvent_t in = nullptr, done = nullptr;
        if ((e = cudaEventCreateWithFlags(&in, cudaEventDisableTiming)) != cudaSuccess) break;
        if ((e = cudaEventCreateWithFlags(&done, cudaEventDisableTiming)) != cudaSuccess) {
            cudaEventDestroy(in);
            break;
        }
        if ((e = cudaMemcpyAsync(const_cast<float *>(plan->x) + ox, x_host + ox, nx, cudaMemcpyHostToDevice, h2d)) ==
                cudaSuccess &&
            (e = cudaMemcpyAsync(const_cast<float *>(plan->dv) + ov, d_dv_host + ov, nv, cudaMemcpyHostToDevice,
                                 h2d)) == cudaSuccess &&
            (e = cudaMemcpyAsync(plan->du + ov, d_u_host + ov, nv, cudaMemcpyHostToDevice, h2d)) == cudaSuccess &&
            (e = cudaEventRecord(in, h2d)) == cudaSuccess && (e = cudaStreamWaitEvent(compute, in, 0)) == cudaSuccess) {
            for (int64_t k = 0; k < cnt && rc == SDM_GX_OK; ++k, ti += step) rc = launch(plan->launch, ti, compute, 0);
            if (rc == SDM_GX_OK && (e = cudaEventRecord(done, compute)) == cudaSuccess &&
                (e = cudaStreamWaitEvent(d2h, done, 0)) == cudaSuccess)
                e = cudaMemcpyAsync(d_u_host + ov, plan->du + ov, nv, cudaMemcpyDeviceToHost, d2h);
        }
        cudaEventDestroy(in);     // released once the pending work that uses it has completed
        cudaEventDestroy(done);
    }
    if (rc != SDM_GX_OK) return rc;
    return e == cudaSuccess ? SDM_GX_OK : fail_cuda(e);
}

int sdm_gx_gemm_plan_set_trace(sdm_gx_plan *plan, unsigned long long *buf, int64_t launches, int32_t *ctas) {
    int rc = plan_check(plan);
    if (rc != SDM_GX_OK) return rc;
#ifndef SDMGX_TRACE
    (void)buf;
    (void)launches;
    (void)ctas;
    return SDM_GX_E_UNSUPPORTED;   // the kernels of this build carry no stamps
#endif
    Launch &l = plan->launch;
    if (l.path != 1 || tma_config(l.config).kind == 1) return SDM_GX_E_UNSUPPORTED;
    if (launches < 0 || launches > kTwo31 / (4 * static_cast<int64_t>(l.grid))) return SDM_GX_E_RANGE;
    if (buf != nullptr && launches > 0) {
        if (reinterpret_cast<uintptr_t>(buf) & 7u) return SDM_GX_E_ALIGN;
        cudaPointerAttributes at{};
        cudaError_t e = cudaPointerGetAttributes(&at, buf);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return SDM_GX_E_DEVICE;
        }
        if ((at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) || at.device != l.device)
            return SDM_GX_E_DEVICE;
        l.tma.trace = buf;
        l.tma.trace_launches = static_cast<int32_t>(launches);
    } else {
        l.tma.trace = nullptr;
        l.tma.trace_launches = 0;
    }
    if (ctas != nullptr) *ctas = l.grid;
    return SDM_GX_OK;
}

int sdm_gx_gemm_plan_geometry(const sdm_gx_plan *plan, sdm_gx_geom *out) {
    if (out == nullptr) return SDM_GX_E_NULL;
    if (plan == nullptr || plan->magic != kPlanMagic || plan->self != plan) return SDM_GX_E_PLAN;
    *out = plan->launch.geom;
    return SDM_GX_OK;
}

void sdm_gx_gemm_plan_destroy(sdm_gx_plan *plan) {
    if (plan == nullptr || plan->magic != kPlanMagic || plan->self != plan) return;
    plan->magic = 0;
    plan->self = nullptr;
    std::free(plan);
}

}  // extern "C"

// ---- the entry point that allocates nothing --------------------------------------------------------------------------
// Its scratch is one static device array per device (each device's module instance has its own copy), used as the
// stream kernel's workspace: partial sums for up to kNoAllocMaxSms CTAs of 128 x 128 tiles, then flags, then launch
// counters. The flags and counters sit at that fixed offset whatever the tile shape. Every launch on the array must
// count the same CTAs, or the per-CTA launch counters drift apart (a hand-off would then wait for a flag that is never
// written, or accept a stale one): build_launch is given stream_ctas_only = the SM count, which admits only stream
// configurations that split a step over exactly one CTA per SM, and a device with more than kNoAllocMaxSms SMs is
// refused. No call allocates; every call shares the array.
namespace {
constexpr int kNoAllocMaxSms = 160;
constexpr size_t kNoAllocWords = (static_cast<size_t>(kNoAllocMaxSms) * 4 + 255) / 256 * 256;
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(kNoAllocMaxSms) * 128 * 128 * 4 + 2 * kNoAllocWords;
static __device__ __align__(256) unsigned char g_sdm_gx_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocState {
    bool init = false;
    void *scratch = nullptr;
};
NoAllocState g_noalloc[kMaxDevices];

// once per device, under the lock: the array's device address, and its flags and launch counters set to zero (a
// memset of existing memory, then a device synchronisation so that every stream sees it). That set-up cannot be part
// of a stream capture, so a first call made while `stream` is being captured is refused.
int noalloc_scratch(int dev, cudaStream_t stream, void **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    NoAllocState &st = g_noalloc[dev];
    if (!st.init) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(stream, &cs);
        if (e != cudaSuccess) return fail_cuda(e);
        if (cs != cudaStreamCaptureStatusNone) return SDM_GX_E_CAPTURE;
        void *a = nullptr;
        e = cudaGetSymbolAddress(&a, g_sdm_gx_noalloc_scratch);
        if (e != cudaSuccess) return fail_cuda(e);
        unsigned char *ctl = static_cast<unsigned char *>(a) + kNoAllocScratchBytes - 2 * kNoAllocWords;
        if ((e = cudaMemset(ctl, 0, 2 * kNoAllocWords)) != cudaSuccess || (e = cudaDeviceSynchronize()) != cudaSuccess)
            return fail_cuda(e);
        st.scratch = a;
        st.init = true;
    }
    *out = st.scratch;
    return SDM_GX_OK;
}
}  // namespace

extern "C" {

int sdm_gx_gemm_step_noalloc(float *d_u, const float *x, const float *d_dv, int64_t ti, int64_t P, int64_t C,
                             int64_t hd, cudaStream_t stream, int pdl) {
    if (d_u == nullptr || x == nullptr || d_dv == nullptr) return SDM_GX_E_NULL;
    if (C < 1 || C > 256 || hd < 1 || hd >= (int64_t(1) << 20)) return SDM_GX_E_SHAPE;
    if (P < 1 || P >= kTwo31 || ti < 0 || ti > (kTwo31 - 1) / P - 1) return SDM_GX_E_RANGE;
    Shape sh{(ti + 1) * P, P, C, hd, contiguous(C, hd)};
    int rc = validate(d_u, x, d_dv, sh, ti * P, (ti + 1) * P);
    if (rc != SDM_GX_OK) return rc;
    int dev = 0;
    const DevState *dsp = nullptr;
    rc = device_state(&dev, &dsp);
    if (rc != SDM_GX_OK) return rc;
    // the array holds the workspace of at most kNoAllocMaxSms CTAs: a larger device is refused, not served slower
    if (dsp->sms > kNoAllocMaxSms) return SDM_GX_E_RANGE;
    void *scratch = nullptr;
    rc = noalloc_scratch(dev, stream, &scratch);
    if (rc != SDM_GX_OK) return rc;
    Launch l;
    rc = build_launch(d_u, x, d_dv, sh, ti * P, P, 0u, &l, scratch, kNoAllocScratchBytes,
                      kNoAllocScratchBytes - 2 * kNoAllocWords, dsp->sms);
    if (rc != SDM_GX_OK) return rc;
    return launch(l, ti, stream, pdl);
}

// the launch sdm_gx_gemm_step_noalloc would make for a step of this shape (for sdm_gx_gemm_geometry; no set-up of
// the array: only its address, which the geometry does not depend on)
int noalloc_geometry(float *d_u, const float *x, const float *d_dv, const Shape &sh, Launch *l) {
    int dev = 0;
    const DevState *dsp = nullptr;
    int rc = device_state(&dev, &dsp);
    if (rc != SDM_GX_OK) return rc;
    if (dsp->sms > kNoAllocMaxSms) return SDM_GX_E_RANGE;
    void *a = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&a, g_sdm_gx_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda(e);
    return build_launch(d_u, x, d_dv, sh, 0, sh.P, 0u, l, a, kNoAllocScratchBytes,
                        kNoAllocScratchBytes - 2 * kNoAllocWords, dsp->sms);
}

int sdm_gx_producer_step(float *d_dv, const float *S, int64_t ti, int64_t P, int64_t C, int64_t hd,
                         cudaStream_t stream, int pdl) {
    if (d_dv == nullptr || S == nullptr) return SDM_GX_E_NULL;
    if (C < 1 || C > 256 || hd < 1 || hd >= (int64_t(1) << 20)) return SDM_GX_E_SHAPE;
    if (P < 1 || P >= kTwo31 || ti < 0 || ti > (kTwo31 - 1) / P - 1) return SDM_GX_E_RANGE;
    if ((reinterpret_cast<uintptr_t>(d_dv) | reinterpret_cast<uintptr_t>(S)) & 3u) return SDM_GX_E_ALIGN;
    const int64_t per_step = P * C * hd;
    const Span a = span_of(d_dv, ti * P, (ti + 1) * P, C * hd, hd, C, hd);
    const Span b = span_of(S, ti * P, (ti + 1) * P, C * hd, hd, C, hd);
    if (overlaps(a, b)) return SDM_GX_E_OVERLAP;
    int dev = 0;
    const DevState *d = nullptr;
    int rc = device_state(&dev, &d);
    if (rc != SDM_GX_OK) return rc;
    cudaError_t e = producer_launch(d_dv, S, ti * per_step, per_step, static_cast<int>(ti & 1), stream, pdl, d->sms);
    if (e != cudaSuccess) return fail_cuda(e);
    g_count_producer.fetch_add(1, std::memory_order_relaxed);
    if (pdl) g_count_pdl.fetch_add(1, std::memory_order_relaxed);
    return SDM_GX_OK;
}

int sdm_gx_gemm_kernel_attrs(int32_t path, int32_t config, int64_t out[4]) {
    if (out == nullptr) return SDM_GX_E_NULL;
    const void *fn = nullptr;
    if (path == 1 && config >= 0 && config < tma_num_configs()) fn = tma_kernel(config);
    if (path == 0 && config >= 0 && config < generic_num_configs()) fn = generic_kernel(config);
    if (fn == nullptr) return SDM_GX_E_FLAGS;
    cudaFuncAttributes a{};
    cudaError_t e = cudaFuncGetAttributes(&a, fn);
    if (e != cudaSuccess) return fail_cuda(e);
    out[0] = a.numRegs;
    out[1] = static_cast<int64_t>(a.localSizeBytes);
    out[2] = static_cast<int64_t>(a.sharedSizeBytes);
    out[3] = a.maxThreadsPerBlock;
    return SDM_GX_OK;
}

int sdm_gx_gemm_config_info(int32_t path, int32_t config, int32_t out[8]) {
    if (out == nullptr) return SDM_GX_E_NULL;
    const ConfigInfo *ci = nullptr;
    if (path == 1 && config >= 0 && config < tma_num_configs()) ci = &tma_config(config);
    if (path == 0 && config >= 0 && config < generic_num_configs()) ci = &generic_config(config);
    if (ci == nullptr) return SDM_GX_E_FLAGS;
    out[0] = ci->TI;
    out[1] = ci->TC;
    out[2] = ci->KB;
    out[3] = ci->stages;
    out[4] = ci->threads;
    out[5] = ci->smem;
    out[6] = path == 1 ? (ci->kind == 3 && ci->shifted ? 4 : ci->kind) : 0;
    out[7] = ci->consumer_warps;
    return SDM_GX_OK;
}

int sdm_gx_gemm_stream_piece(int64_t ntiles, int32_t C, int32_t G, int32_t b, int32_t q, int32_t out[4]) {
    if (out == nullptr) return SDM_GX_E_NULL;
    if (C < 1 || C > 256 || G < 1 || ntiles < G || ntiles >= kTwo31 || b < 0 || b >= G) return SDM_GX_E_RANGE;
    const Pieces R = cta_pieces(static_cast<int>(ntiles), C, b, G, stream_kappa(ntiles, C, G));
    if (q < 0) return R.count;
    if (q >= R.count) return SDM_GX_E_RANGE;
    const Piece pc = piece_at(R, C, q);
    out[0] = pc.t;
    out[1] = pc.j0;
    out[2] = pc.j1;
    out[3] = pc.kind;
    return SDM_GX_OK;
}

int sdm_gx_gemm_choose_config(int32_t path, int32_t sms, const int32_t *occ, int32_t n_occ, int32_t slab_ok,
                              int64_t P, int64_t C, int64_t hd, size_t ws_bytes) {
    if (occ == nullptr) return SDM_GX_E_NULL;
    if (path != 0 && path != 1) return SDM_GX_E_FLAGS;
    if (C < 1 || C > 256 || hd < 1 || hd >= (int64_t(1) << 20)) return SDM_GX_E_SHAPE;
    const int nk = path == 1 ? tma_num_configs() : generic_num_configs();
    if (sms < 1 || sms > 4096 || n_occ != nk || P < 1 || P >= kTwo31) return SDM_GX_E_RANGE;
    DevState d;
    d.sms = sms;
    d.slab_ok = slab_ok != 0;
    for (int k = 0; k < nk; ++k) {
        if (occ[k] < 0) return SDM_GX_E_RANGE;
        (path == 1 ? d.tma_occ : d.gen_occ)[k] = occ[k];
    }
    if (path == 0) return choose_generic_config(d, P, C, hd, -1);
    const int k = choose_tma_config(d, P, C, hd, -1, ws_bytes, 0);
    return k >= 0 ? k : SDM_GX_E_SMEM;
}

int sdm_gx_gemm_num_configs(int32_t path) {
    if (path == 1) return tma_num_configs();
    if (path == 0) return generic_num_configs();
    return 0;
}

int sdm_gx_device_error(uint32_t *word, int clear) {
    if (word == nullptr) return SDM_GX_E_NULL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e);
    uint32_t w = 0;
    if ((e = cudaMemcpyFromSymbol(&w, g_sdm_gx_error_word, sizeof(w))) != cudaSuccess) return fail_cuda(e);
    *word = w;
    if (clear) {
        const uint32_t z = 0;
        if ((e = cudaMemcpyToSymbol(g_sdm_gx_error_word, &z, sizeof(z))) != cudaSuccess) return fail_cuda(e);
    }
    return (w & kErrFatalMask) ? SDM_GX_E_DEVICE_FAULT : SDM_GX_OK;   // a recomputed hand-off alone is no fault
}

void sdm_gx_launch_counts(int64_t out[4]) {
    if (out == nullptr) return;
    out[0] = g_count_step.load();
    out[1] = g_count_producer.load();
    out[2] = g_count_pdl.load();
    out[3] = g_count_succ.load();
}

int sdm_gx_last_cuda_error(void) { return t_last_cuda; }

const char *sdm_gx_strerror(int status) {
    switch (status) {
        case SDM_GX_OK: return "ok";
        case SDM_GX_E_NULL: return "a required pointer is NULL";
        case SDM_GX_E_SHAPE: return "need 1 <= C <= 256 and 1 <= hd < 2^20";
        case SDM_GX_E_RANGE: return "step out of range (need 1 <= P <= N < 2^31 and 0 <= ti < N / P)";
        case SDM_GX_E_ALIGN: return "operands must be 4-byte aligned (a plan workspace 256-byte aligned)";
        case SDM_GX_E_OVERLAP: return "d_u overlaps x or d_dv (the in-place update needs disjoint operands), or the workspace overlaps an operand";
        case SDM_GX_E_STRIDE: return "strides do not describe a non-overlapping [N, rows, cols] layout";
        case SDM_GX_E_GRID: return "too many tiles in one step";
        case SDM_GX_E_SMEM: return "shared memory exceeds the device's opt-in limit";
        case SDM_GX_E_DEVICE: return "operands must be device memory of the current device";
        case SDM_GX_E_PLAN: return "plan is NULL or corrupt";
        case SDM_GX_E_PLAN_TI: return "step outside [0, ti_max] of the plan";
        case SDM_GX_E_PLAN_DEVICE: return "the current device is not the plan's device";
        case SDM_GX_E_FLAGS: return "unknown flags or invalid forced configuration";
        case SDM_GX_E_CUDA: return "a CUDA runtime call failed (see sdm_gx_last_cuda_error)";
        case SDM_GX_E_DEVICE_FAULT: return "a kernel gave up a bounded wait (device error word set)";
        case SDM_GX_E_UNSUPPORTED: return "the current device is not an sm_103 GPU, or the plan's kernel cannot do this (a timeline on the generic or slab kernel)";
        case SDM_GX_E_ALLOC: return "host allocation failed";
        case SDM_GX_E_CAPTURE: return "the first sdm_gx_gemm_step_noalloc call on a device sets up its static workspace and cannot run while the stream is being captured";
        default: return "unknown status";
    }
}

}  // extern "C"
