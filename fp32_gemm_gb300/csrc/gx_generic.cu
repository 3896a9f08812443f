// The generic kernel of the gx_gemm step update (any element strides, 4-byte alignment, any C <= 256 and hd), and
// the synthetic producer kernel of the chained workload. sm_103a.
//
// Generic kernel: CTAs of 256 threads loop over tiles of TI rows x 64 columns of one chunk (grid <= resident slots);
// a large-tile variant (below) serves steps whose 128 x 64 tiles fill the SMs. x may be given transposed (stored as
// [n][i][j], x_si > 1): the small-tile kernel stages it with j fastest, so that its global reads stay coalesced.
// Thread (tx, ty) of a 16 x 16 layout owns rows i0 + ty + 16 r (r < TI / 16) and columns c0 + tx + 16 q (q < 4), so
// global reads and writes of d_u are coalesced along c. The j range is staged KB = 32 rows at a time into shared
// memory (xs[KB][TI] from x[n, j, i], ds[KB][64] from d_dv[n, j, c], zero past C / hd) with plain loads, and every
// output runs the chain acc = fmaf(x[n,j,i], d_dv[n,j,c], acc), j = 0..C-1 in order from +0, then d_u + acc
// (sparse_delta_memory/cuda/gx_gemm_cuda.py, module docstring formula and gx_gemm_kernel).
// Programmatic dependent launch: the first tile's d_u values are read into registers before griddepcontrol.wait;
// x, d_dv are read and d_u written after it.
#include "gx_device.cuh"
#include "gx_internal.h"

namespace sdmgx {
namespace {

constexpr int kGenTC = 64, kGenKB = 32, kGenNT = 256, kGenTX = 16, kGenTY = 16, kGenRC = kGenTC / kGenTX;

template <int TI>
__global__ void __launch_bounds__(kGenNT) gx_generic_kernel(const GenericParams p) {
    constexpr int RI = TI / kGenTY;
    __shared__ float xs[kGenKB][TI + 1];   // + 1: the transposed staging writes columns of it without bank conflicts
    __shared__ float ds[kGenKB][kGenTC];
    const int tx = static_cast<int>(threadIdx.x) % kGenTX;
    const int ty = static_cast<int>(threadIdx.x) / kGenTX;
    const int per_chunk = p.nib * p.ncb;
    bool waited = false;
    for (int t = static_cast<int>(blockIdx.x); t < p.ntiles; t += static_cast<int>(gridDim.x)) {
        const int pp = t / per_chunk;
        const int rem = t - pp * per_chunk;
        const int ib = rem / p.ncb;
        const int cb = rem - ib * p.ncb;
        const int64_t n = p.n_base + pp;
        const int i0 = ib * TI, c0 = cb * kGenTC;
        const float *xn = p.x + n * p.x_sn;
        const float *dvn = p.dv + n * p.dv_sn;
        float *dun = p.du + n * p.du_sn;
        float u[RI][kGenRC];
#pragma unroll
        for (int r = 0; r < RI; ++r) {
            const int i = i0 + ty + kGenTY * r;
#pragma unroll
            for (int q = 0; q < kGenRC; ++q) {
                const int c = c0 + tx + kGenTX * q;
                u[r][q] = (i < p.C && c < p.hd) ? dun[static_cast<int64_t>(i) * p.du_si + c] : 0.0f;
            }
        }
        if (!waited) {
            dev::grid_dependency_wait();
            dev::launch_dependents();
            waited = true;
        }
        float acc[RI][kGenRC];
#pragma unroll
        for (int r = 0; r < RI; ++r) {
#pragma unroll
            for (int q = 0; q < kGenRC; ++q) acc[r][q] = 0.0f;
        }
        for (int j0 = 0; j0 < p.C; j0 += kGenKB) {
            const int nj = (p.C - j0) < kGenKB ? (p.C - j0) : kGenKB;
            __syncthreads();   // the previous block's reads are done before the buffers are overwritten
            if (p.x_si == 1) {   // x[n, j, i0 .. i0 + TI - 1] rows: i fastest
                for (int e = static_cast<int>(threadIdx.x); e < kGenKB * TI; e += kGenNT) {
                    const int jj = e / TI, ii = e - jj * TI;
                    xs[jj][ii] =
                        (jj < nj && i0 + ii < p.C) ? xn[static_cast<int64_t>(j0 + jj) * p.x_sj + i0 + ii] : 0.0f;
                }
            } else {             // x stored transposed: j fastest along the stored rows i
                for (int e = static_cast<int>(threadIdx.x); e < kGenKB * TI; e += kGenNT) {
                    const int ii = e / kGenKB, jj = e - ii * kGenKB;
                    xs[jj][ii] = (jj < nj && i0 + ii < p.C)
                                     ? xn[static_cast<int64_t>(i0 + ii) * p.x_si + static_cast<int64_t>(j0 + jj) * p.x_sj]
                                     : 0.0f;
                }
            }
            for (int e = static_cast<int>(threadIdx.x); e < kGenKB * kGenTC; e += kGenNT) {
                const int jj = e / kGenTC, cc = e - jj * kGenTC;
                ds[jj][cc] =
                    (jj < nj && c0 + cc < p.hd) ? dvn[static_cast<int64_t>(j0 + jj) * p.dv_sj + c0 + cc] : 0.0f;
            }
            __syncthreads();
            for (int jj = 0; jj < nj; ++jj) {
                float d[kGenRC];
#pragma unroll
                for (int q = 0; q < kGenRC; ++q) d[q] = ds[jj][tx + kGenTX * q];
#pragma unroll
                for (int r = 0; r < RI; ++r) {
                    const float xv = xs[jj][ty + kGenTY * r];
#pragma unroll
                    for (int q = 0; q < kGenRC; ++q) acc[r][q] = fmaf(xv, d[q], acc[r][q]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RI; ++r) {
            const int i = i0 + ty + kGenTY * r;
            if (i >= p.C) continue;
#pragma unroll
            for (int q = 0; q < kGenRC; ++q) {
                const int c = c0 + tx + kGenTX * q;
                if (c < p.hd) dun[static_cast<int64_t>(i) * p.du_si + c] = __fadd_rn(u[r][q], acc[r][q]);
            }
        }
    }
    if (!waited) {   // a CTA without a tile still orders itself after the predecessor
        dev::grid_dependency_wait();
        dev::launch_dependents();
    }
}

template <int TI>
cudaError_t launch_generic(const GenericParams &p, int grid, cudaStream_t st, int pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kGenNT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gx_generic_kernel<TI>, p);
}

template <int TI>
ConfigInfo generic_info() {
    return ConfigInfo{TI, kGenTC, kGenKB, 1, kGenNT, 0, TI / kGenTY, kGenRC, kGenNT / 32, 40, 0};
}

// Large-tile generic kernel, for steps whose 128 x 64 tiles fill the SMs. CTAs of 256 threads loop over 128 x 64
// tiles. Warp w owns rows 32 (w % 4) .. + 31 and columns 32 (w / 4) .. + 31 in lanes of 4 x 8; a thread owns rows
// ro .. ro + 3 and ro + 16 .. ro + 19 (ro = 32 (w % 4) + 4 (lane / 8)) of columns co .. co + 3 (co = 32 (w / 4) +
// 4 (lane % 8)), as in the TMA kernel's consumers, and runs its 8 x 4 chains with packed FMAs along rows (lane by lane
// the same fused multiply-add as fmaf). j is staged 32 rows at a time into one of two shared buffers by 4-byte
// asynchronous copies (cp.async: any strides, zero fill past C / hd); the copies of the next block, of this tile or of
// the CTA's next tile, are in flight while the current block is used. d_u is prefetched into L2 when a tile starts, read
// in the epilogue and written as d_u + acc; every access comes after the dependency wait.
constexpr int kBigTI = 128, kBigTC = 64, kBigKB = 32, kBigNT = 256;
constexpr int kBigXE = kBigKB * kBigTI / kBigNT;   // x elements a thread copies per block of j (rows xj + 2k)
constexpr int kBigDE = kBigKB * kBigTC / kBigNT;   // d_dv elements (rows dj + 4k)

// 4-byte asynchronous copy global -> shared (cached in L1); src_bytes = 0 writes a zero and reads nothing
__device__ __forceinline__ void cp_async_4(uint32_t dst, const float *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most N of this thread's copy groups are still in flight
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(ptr)));
}

__device__ __forceinline__ void big_chain_j(const float *xb, const float *db, int jj, int ro, int co,
                                            float (&acc)[8][4]) {
    float a[8], b[4];
    dev::Vec<4>::load(xb + jj * kBigTI + ro, a);
    dev::Vec<4>::load(xb + jj * kBigTI + ro + 16, a + 4);
    dev::Vec<4>::load(db + jj * kBigTC + co, b);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int r = 0; r < 8; r += 2) dev::fma2(acc[r][c], acc[r + 1][c], a[r], a[r + 1], b[c], b[c]);
    }
}

__global__ void __launch_bounds__(kBigNT, 2) gx_generic_big_kernel(const GenericParams p) {
    __shared__ __align__(16) float xs[2][kBigKB][kBigTI];
    __shared__ __align__(16) float ds[2][kBigKB][kBigTC];
    const int tid = static_cast<int>(threadIdx.x);
    const int warp = tid / 32, lane = tid % 32;
    const int ro = (warp % 4) * 32 + (lane / 8) * 4;
    const int co = (warp / 4) * 32 + (lane % 8) * 4;
    const int xi = tid % kBigTI, xj = tid / kBigTI;
    const int di = tid % kBigTC, dj = tid / kBigTC;
    const int per_chunk = p.nib * p.ncb;
    const int nkb = (p.C + kBigKB - 1) / kBigKB;
    const int stride = static_cast<int>(gridDim.x);
    dev::grid_dependency_wait();
    dev::launch_dependents();
    const uint32_t xs_s = dev::smem_addr(&xs[0][0][0]);
    const uint32_t ds_s = dev::smem_addr(&ds[0][0][0]);
    // this thread's copies of block kb (rows j0 .. j0 + 31) of tile t into buffer b, as one copy group
    auto issue = [&](int t, int kb, int b) {
        const int pp = t / per_chunk;
        const int rem = t - pp * per_chunk;
        const int ib = rem / p.ncb;
        const int64_t n = p.n_base + pp;
        const int i0 = ib * kBigTI, c0 = (rem - ib * p.ncb) * kBigTC;
        const float *xn = p.x + n * p.x_sn;
        const float *dvn = p.dv + n * p.dv_sn;
        const int j0 = kb * kBigKB;
#pragma unroll
        for (int k = 0; k < kBigXE; ++k) {
            const int j = j0 + xj + 2 * k, i = i0 + xi;
            const bool ok = j < p.C && i < p.C;
            cp_async_4(xs_s + static_cast<uint32_t>(((b * kBigKB + xj + 2 * k) * kBigTI + xi) * 4),
                            ok ? xn + static_cast<int64_t>(j) * p.x_sj + i : xn, ok ? 4u : 0u);
        }
#pragma unroll
        for (int k = 0; k < kBigDE; ++k) {
            const int j = j0 + dj + 4 * k, c = c0 + di;
            const bool ok = j < p.C && c < p.hd;
            cp_async_4(ds_s + static_cast<uint32_t>(((b * kBigKB + dj + 4 * k) * kBigTC + di) * 4),
                            ok ? dvn + static_cast<int64_t>(j) * p.dv_sj + c : dvn, ok ? 4u : 0u);
        }
        cp_async_commit();
    };
    int s = 0;   // blocks this CTA has used so far; block s sits in buffer s & 1
    if (static_cast<int>(blockIdx.x) < p.ntiles) issue(static_cast<int>(blockIdx.x), 0, 0);
    for (int t = static_cast<int>(blockIdx.x); t < p.ntiles; t += stride) {
        const int pp = t / per_chunk;
        const int rem = t - pp * per_chunk;
        const int ib = rem / p.ncb;
        const int64_t n = p.n_base + pp;
        const int i0 = ib * kBigTI, c0 = (rem - ib * p.ncb) * kBigTC;
        float *dun = p.du + n * p.du_sn;
        if (c0 + co < p.hd) {   // the epilogue's d_u rows into L2 while the chain runs
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = i0 + ro + (r / 4) * 16 + (r % 4);
                if (i < p.C) prefetch_l2(dun + static_cast<int64_t>(i) * p.du_si + c0 + co);
            }
        }
        float acc[8][4];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[r][c] = 0.0f;   // +0: the chain's start value
        }
        for (int kb = 0; kb < nkb; ++kb, ++s) {
            // the next block (of this tile, else block 0 of the CTA's next tile) goes into the other buffer, which
            // every thread left at the barrier that ended the previous block
            const int nt = kb + 1 < nkb ? t : t + stride;
            if (nt < p.ntiles) {
                issue(nt, kb + 1 < nkb ? kb + 1 : 0, (s + 1) & 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();   // every thread's copies of block s have landed
            const float *xb = &xs[s & 1][0][0];
            const float *db = &ds[s & 1][0][0];
            const int nj = p.C - kb * kBigKB < kBigKB ? p.C - kb * kBigKB : kBigKB;
            if (nj == kBigKB) {
#pragma unroll 8
                for (int jj = 0; jj < kBigKB; ++jj) big_chain_j(xb, db, jj, ro, co, acc);
            } else {
#pragma unroll 1
                for (int jj = 0; jj < nj; ++jj) big_chain_j(xb, db, jj, ro, co, acc);
            }
            __syncthreads();   // buffer s & 1 is free for block s + 2
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int i = i0 + ro + (r / 4) * 16 + (r % 4);
            if (i >= p.C) continue;
            float *row = dun + static_cast<int64_t>(i) * p.du_si;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int cc = c0 + co + c;
                if (cc < p.hd) row[cc] = __fadd_rn(row[cc], acc[r][c]);
            }
        }
    }
}

cudaError_t launch_generic_big(const GenericParams &p, int grid, cudaStream_t st, int pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kBigNT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gx_generic_big_kernel, p);
}

struct GEntry {
    ConfigInfo info;
    const void *fn;
    cudaError_t (*launch)(const GenericParams &, int, cudaStream_t, int);
};
// the large-tile kernel stays last (the host's choice relies on it)
const GEntry kGen[] = {
    {generic_info<16>(), reinterpret_cast<const void *>(&gx_generic_kernel<16>), &launch_generic<16>},
    {generic_info<32>(), reinterpret_cast<const void *>(&gx_generic_kernel<32>), &launch_generic<32>},
    {generic_info<64>(), reinterpret_cast<const void *>(&gx_generic_kernel<64>), &launch_generic<64>},
    {ConfigInfo{kBigTI, kBigTC, kBigKB, 2, kBigNT, 0, 8, 4, kBigNT / 32, 50, 0},   // 48 KB of static shared memory
     reinterpret_cast<const void *>(&gx_generic_big_kernel), &launch_generic_big},
};

// ---- synthetic producer: d_dv[base + e] = +-S[base + e], e < count --------------------------------------------------
// The first grid-wide pass of S is read before griddepcontrol.wait; every write of d_dv comes after it.
constexpr int kProdNT = 256;

__global__ void __launch_bounds__(kProdNT) gx_producer_kernel(float *__restrict__ dv, const float *__restrict__ S,
                                                               int64_t base, int64_t count, uint32_t flip, int vec) {
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * kProdNT;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kProdNT + threadIdx.x;
    if (vec) {
        const float4 *src = reinterpret_cast<const float4 *>(S + base);
        float4 *dst = reinterpret_cast<float4 *>(dv + base);
        const int64_t nv = count / 4;
        float4 v = tid < nv ? src[tid] : make_float4(0.f, 0.f, 0.f, 0.f);
        dev::grid_dependency_wait();
        dev::launch_dependents();
        for (int64_t e = tid; e < nv; e += nthr) {
            if (e != tid) v = src[e];
            uint4 b = *reinterpret_cast<uint4 *>(&v);
            b.x ^= flip;
            b.y ^= flip;
            b.z ^= flip;
            b.w ^= flip;
            dst[e] = *reinterpret_cast<float4 *>(&b);
        }
    } else {
        float v = tid < count ? S[base + tid] : 0.0f;
        dev::grid_dependency_wait();
        dev::launch_dependents();
        for (int64_t e = tid; e < count; e += nthr) {
            if (e != tid) v = S[base + e];
            dv[base + e] = __uint_as_float(__float_as_uint(v) ^ flip);
        }
    }
}

// ---- synthetic successor: a consumer of d_u(ti) that runs right after the step under PDL ----------------------------
// One warp per chunk n of step ti reads the chunk's leading row d_u[n, 0, :] and writes out[n] = its sum in a fixed
// order: lane l adds d_u[n, 0, l], d_u[n, 0, l + 32], ... left to right from +0, then the 32 partial sums are combined
// by an xor butterfly (offsets 16, 8, 4, 2, 1), one rounding per add; lane 0's value is stored. The kernel triggers
// its dependents first (so the next step's prologue may overlap it), then waits for the step that wrote d_u(ti).
constexpr int kSuccNT = 256;

__global__ void __launch_bounds__(kSuccNT) gx_successor_kernel(const float *__restrict__ du, float *__restrict__ out,
                                                                int64_t n0, int32_t P, int32_t hd, int64_t du_sn) {
    dev::launch_dependents();
    dev::grid_dependency_wait();
    const int lane = static_cast<int>(threadIdx.x) % 32;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kSuccNT / 32);
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * (kSuccNT / 32) + threadIdx.x / 32; p < P; p += warps) {
        const float *row = du + (n0 + p) * du_sn;
        float v = 0.0f;
        for (int c = lane; c < hd; c += 32) v = __fadd_rn(v, row[c]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
        if (lane == 0) out[n0 + p] = v;
    }
}

}  // namespace

cudaError_t successor_launch(const float *du, float *out, int64_t n0, int P, int hd, int64_t du_sn, cudaStream_t st,
                             int pdl, int sms) {
    int64_t blocks = (static_cast<int64_t>(P) + kSuccNT / 32 - 1) / (kSuccNT / 32);
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kSuccNT);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gx_successor_kernel, du, out, n0, P, hd, du_sn);
}

int generic_num_configs() { return static_cast<int>(sizeof(kGen) / sizeof(kGen[0])); }
const ConfigInfo &generic_config(int k) { return kGen[k].info; }
const void *generic_kernel(int k) { return kGen[k].fn; }
cudaError_t generic_launch(int k, const GenericParams &p, int grid, cudaStream_t st, int pdl) {
    return kGen[k].launch(p, grid, st, pdl);
}

cudaError_t producer_launch(float *dv, const float *S, int64_t base, int64_t count, int negate, cudaStream_t st,
                            int pdl, int sms) {
    if (count <= 0) return cudaSuccess;
    const int vec = ((reinterpret_cast<uintptr_t>(dv + base) | reinterpret_cast<uintptr_t>(S + base)) & 15u) == 0 &&
                    (count % 4) == 0;
    const int64_t units = vec ? count / 4 : count;
    int64_t blocks = (units + kProdNT - 1) / kProdNT;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kProdNT);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gx_producer_kernel, dv, S, base, count, negate ? 0x80000000u : 0u, vec);
}

}  // namespace sdmgx
