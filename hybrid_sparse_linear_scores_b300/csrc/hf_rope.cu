// hf_rope.cu -- the relative temporal RoPE pre-step (Hybrid Forcing, English
// technical summary, section 2.C "Stability Enhancements": temporal RoPE
// indices are kept under one fixed upper bound in training and inference,
// positions taken as relative offsets).
//
// Rotary embedding (RoFormer) on channel pairs (2i, 2i+1), i < rot_dims/2:
// angle p * base^(-2i/rot_dims), where p is the frame's offset inside the
// current window clamped to [0, max_offset]; channels >= rot_dims are copied.
// Every token of a frame shares its angles, so a CTA (one frame of one head,
// 64 tokens) forms the frame's cos/sin table once in shared memory.  One
// 16-byte load and one 16-byte store per 8 channels, a thread's loads all
// issued before its stores: bound by HBM.
#include <cuda_runtime.h>

#include <cstdint>

#include "hf_internal.h"
#include "hf_ptx.cuh"

namespace hf {
namespace {

constexpr int kRopeTokens = 64;    // tokens per CTA
constexpr int kRopeThreads = 256;

__global__ void __launch_bounds__(kRopeThreads) rope_kernel(const RopeParams p)
{
    __shared__ float2 cs[64];                    // (cos, sin) per channel pair (d <= 128)
    const int hf = blockIdx.y;                   // head * n_frames + frame
    const int h = hf / p.n_frames;
    const int f = hf - h * p.n_frames;
    const float pos = (float)p.pos[f];
    for (int i = threadIdx.x; i < p.rot_dims / 2; i += blockDim.x) {
        float s, c;
        sincosf(pos * p.inv_freq[i], &s, &c);
        cs[i] = make_float2(c, s);
    }
    __syncthreads();
    const int chunks = p.d / 8;                  // 16-byte chunks per token
    const size_t base = (size_t)h * p.head_stride + (size_t)p.slot[f] * p.frame_stride;
    const int t0 = blockIdx.x * kRopeTokens;
    const int n_items = min(kRopeTokens, p.nf - t0) * chunks;
    // every load of the thread is issued before any store (bytes in flight)
    constexpr int kPer = kRopeTokens * 16 / kRopeThreads;   // items per thread at d = 128
    for (int i0 = threadIdx.x; i0 < n_items; i0 += kRopeThreads * kPer) {
        uint4 v[kPer];
        size_t off[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int it = i0 + k * kRopeThreads;
            const int t = t0 + it / chunks;
            const int ch = it - (it / chunks) * chunks;
            off[k] = base + (size_t)t * p.d + ch * 8;
            if (it < n_items) v[k] = *reinterpret_cast<const uint4*>(p.src + off[k]);
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int it = i0 + k * kRopeThreads;
            if (it >= n_items) break;
            const int ch = it % chunks;
            if (ch * 8 < p.rot_dims) {           // rot_dims is a multiple of 8
                uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 r = cs[ch * 4 + j];
                    const float x0 = bf16_lo(w[j]), x1 = bf16_hi(w[j]);
                    w[j] = pack_bf16(x0 * r.x - x1 * r.y, x0 * r.y + x1 * r.x);
                }
                v[k] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            *reinterpret_cast<uint4*>(p.dst + off[k]) = v[k];
        }
    }
}

}  // namespace

int launch_rope(const RopeParams& p, void* stream)
{
    const dim3 grid((p.nf + kRopeTokens - 1) / kRopeTokens, p.BH * p.n_frames);
    rope_kernel<<<grid, kRopeThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace hf
