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
// 16-byte load and one 16-byte store per 8 channels: bound by HBM.
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
    for (int it = threadIdx.x; it < n_items; it += blockDim.x) {
        const int t = t0 + it / chunks;
        const int ch = it - (it / chunks) * chunks;
        const size_t off = base + (size_t)t * p.d + ch * 8;
        uint4 v = *reinterpret_cast<const uint4*>(p.src + off);
        if (ch * 8 < p.rot_dims) {               // rot_dims is a multiple of 8
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 r = cs[ch * 4 + k];
                const float x0 = bf16_lo(w[k]), x1 = bf16_hi(w[k]);
                w[k] = pack_bf16(x0 * r.x - x1 * r.y, x0 * r.y + x1 * r.x);
            }
            v = make_uint4(w[0], w[1], w[2], w[3]);
        }
        *reinterpret_cast<uint4*>(p.dst + off) = v;
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
