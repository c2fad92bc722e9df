// hf_linear.cu -- the linear temporal attention read outside the fused
// forward (Hybrid Forcing, English technical summary, section 2.A.1 "Linear
// Temporal Attention"), the state reset, and the bounded-wait self-test
// kernel.  (The fused forward's state operand is prepared by the prologue
// kernel in hf_select.cu.)
#include <cuda_runtime.h>

#include <cstdint>

#include "hf_internal.h"
#include "hf_ptx.cuh"

namespace hf {
namespace {

// Standalone linear read in fp32 on CUDA cores: o = phi(q)^T S / (phi(q)^T z + eps).
// CTA = 256 threads handles ROWS query rows of one head; S and z of the head
// are staged in shared memory; each thread computes 8 output channels of one
// row (D/8 threads per row).
template <int D>
__global__ void __launch_bounds__(256) linear_read_kernel(const uint16_t* __restrict__ Q, const float* __restrict__ S,
                                                          const float* __restrict__ z, Geom g, float* __restrict__ O,
                                                          int accumulate)
{
    constexpr int TPR = D / 8;              // threads per row
    constexpr int RPI = 256 / TPR;          // rows per iteration
    constexpr int ROWS = 128;
    extern __shared__ __align__(16) float sm[];
    float* sS = sm;                         // [D][D]
    float* sz = sS + D * D;                 // [D]
    float* sphi = sz + D;                   // [RPI][D]
    const int nq = g.C * g.nf;
    const int tiles = (nq + ROWS - 1) / ROWS;
    const int bh = blockIdx.x / tiles;
    const int row0 = (blockIdx.x - bh * tiles) * ROWS;
    for (int i = threadIdx.x; i < D * D / 4; i += 256)
        reinterpret_cast<float4*>(sS)[i] = reinterpret_cast<const float4*>(S + (size_t)bh * D * D)[i];
    for (int i = threadIdx.x; i < D; i += 256) sz[i] = z[(size_t)bh * D + i];
    const int rl = threadIdx.x / TPR;
    const int part = threadIdx.x % TPR;
    for (int rb = 0; rb < ROWS; rb += RPI) {
        __syncthreads();
        const int row = row0 + rb + rl;
        if (row < nq) {
            const uint16_t* q = Q + ((size_t)bh * nq + row) * D;
            for (int c = part; c < D; c += TPR) {
                const float x = __uint_as_float((uint32_t)q[c] << 16);
                sphi[rl * D + c] = phi_elu1(x);
            }
        }
        __syncthreads();
        if (row < nq) {
            const float* ph = sphi + rl * D;
            float den = g.eps;
            float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int c = 0; c < D; ++c) {
                const float f = ph[c];
                den = fmaf(f, sz[c], den);
                const float* srow = sS + c * D + part * 8;
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[k] = fmaf(f, srow[k], acc[k]);
            }
            const float inv = 1.0f / den;
            float* o = O + ((size_t)bh * nq + row) * D + part * 8;
#pragma unroll
            for (int k = 0; k < 8; ++k) o[k] = accumulate ? o[k] + acc[k] * inv : acc[k] * inv;
        }
    }
}

__global__ void state_reset_kernel(float* __restrict__ S, float* __restrict__ z, long nS, long nz)
{
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < nS) S[i] = 0.0f;
    if (i < nz) z[i] = 0.0f;
}

// Waits on a barrier that nothing will ever complete, with the given limit.
__global__ void selftest_wait_kernel(uint32_t* status, uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        WaitCtl w{&abort_flag, status, limit_ns};
        (void)mbar_wait(&bar, 0, w, SITE_SELFTEST);
        // release the barrier so no wait is left pending at exit
        mbar_arrive(&bar);
    }
}

}  // namespace

template <int D>
static int launch_lr(const uint16_t* Q, const float* S, const float* z, const Geom& g, float* O, int accumulate,
                     cudaStream_t st)
{
    const size_t bytes = sizeof(float) * (D * D + D + (256 / (D / 8)) * D);
    cudaError_t e = cudaFuncSetAttribute(linear_read_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return (int)e;
    const int nq = g.C * g.nf;
    const int tiles = (nq + 127) / 128;
    linear_read_kernel<D><<<g.BH * tiles, 256, bytes, st>>>(Q, S, z, g, O, accumulate);
    return (int)cudaGetLastError();
}

int launch_linear_read(const uint16_t* Q, const float* S, const float* z, const Geom& g, float* O, int accumulate,
                       void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return g.d == 128 ? launch_lr<128>(Q, S, z, g, O, accumulate, st) : launch_lr<64>(Q, S, z, g, O, accumulate, st);
}

int launch_state_reset(float* S, float* z, const Geom& g, void* stream)
{
    const long nS = (long)g.BH * g.d * g.d, nz = (long)g.BH * g.d;
    state_reset_kernel<<<(unsigned)((nS + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(S, z, nS, nz);
    return (int)cudaGetLastError();
}

int launch_selftest_wait(uint32_t* status, uint64_t limit_ns, void* stream)
{
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
    return (int)cudaGetLastError();
}

}  // namespace hf
