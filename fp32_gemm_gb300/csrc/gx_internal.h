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
};

// Parameters of the generic kernel (any strides, 4-byte alignment).
struct GenericParams {
    float *du;
    const float *x;
    const float *dv;
    int64_t x_sn, x_sj, dv_sn, dv_sj, du_sn, du_si;
    int64_t n_base;
    int32_t P, C, hd;
    int32_t nib, ncb;
    int32_t ntiles;
};

struct ConfigInfo {
    int TI, TC, KB, stages, threads, smem, RM, RN, consumer_warps;
    int eff;    // measured FMA-pipe efficiency (percent) with every SM busy
    int slab;   // 1: the balanced slab kernel (TI = slab rows; needs C % TI == 0 and C / TI >= 3)
};

// TMA path
int tma_num_configs();
const ConfigInfo &tma_config(int k);
const void *tma_kernel(int k);
cudaError_t tma_launch(int k, const TmaParams &p, int grid, cudaStream_t st, int pdl);

// generic path (config k: 16, 32, 64 rows per tile)
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
