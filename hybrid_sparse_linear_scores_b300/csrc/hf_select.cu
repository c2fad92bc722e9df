// hf_select.cu -- block pooling, block importance scores and the top-K block
// selector of the block-sparse sliding-window path (Hybrid Forcing, English
// technical summary, section 2.A.2: block importance scores are computed
// and only the top-K most informative blocks are retained).
//
// The arithmetic is fixed so that scores and indices are bit-reproducible:
//   pooled[ch] = (((x_0 + x_1) + x_2) + ...) / n      float32, RN, token order
//   score      = fma(q[d-1], k[d-1], ... fma(q[0], k[0], 0))  ascending ch
//   score += 0.0f (-0 -> +0)
// Top-K: order by (score desc, block index asc); keep K; write ascending.
//
// All three kernels are HBM- or latency-bound; none touches tensor cores.
#include <cuda_runtime.h>

#include <cstdint>

#include "hf_internal.h"

namespace hf {
namespace {

// ---------------------------------------------------------------------------
// Pooling: one task = one block (beta tokens of one frame) of Q (chunk) or
// K (window, through the ring).  D/8 threads per task, 8 channels each
// (one 16-byte load per token); sequential float32 sums.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) pool_kernel(const uint16_t* __restrict__ Q, const uint16_t* __restrict__ Kc,
                                                   Geom g, SlotMap sm, float* __restrict__ qp,
                                                   float* __restrict__ kp)
{
    constexpr int TPB = D / 8;
    constexpr int TASKS = 256 / TPB;
    const int task = blockIdx.x * TASKS + threadIdx.x / TPB;
    const int part = threadIdx.x % TPB;
    const int per_head = g.nqb + g.nkb;
    if (task >= g.BH * per_head) return;
    const int bh = task / per_head;
    const int b = task - bh * per_head;

    const uint16_t* src;
    float* dst;
    int j;
    if (b < g.nqb) {
        const int c = b / g.bpf;
        j = b - c * g.bpf;
        src = Q + ((size_t)bh * g.C * g.nf + (size_t)c * g.nf + (size_t)j * g.beta) * D;
        dst = qp + ((size_t)bh * g.nqb + b) * D;
    } else {
        const int kb = b - g.nqb;
        const int w = kb / g.bpf;
        j = kb - w * g.bpf;
        const int slot = sm.s[w];
        src = Kc + (((size_t)bh * g.W + slot) * g.slot_stride + (size_t)j * g.beta) * D;
        dst = kp + ((size_t)bh * g.nkb + kb) * D;
    }
    const int n = min(g.beta, g.nf - j * g.beta);
    const uint4* p = reinterpret_cast<const uint4*>(src) + part;
    constexpr int ROW = D / 8;   // uint4 per token row

    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;

    for (int t0 = 0; t0 < n; t0 += 8) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (t0 + u < n) v[u] = __ldg(p + (size_t)(t0 + u) * ROW);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (t0 + u < n) {
                const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = __fadd_rn(acc[2 * i], __uint_as_float(w4[i] << 16));
                    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __uint_as_float(w4[i] & 0xFFFF0000u));
                }
            }
        }
    }
    const float fn = static_cast<float>(n);
    float4 o0, o1;
    o0.x = __fdiv_rn(acc[0], fn);
    o0.y = __fdiv_rn(acc[1], fn);
    o0.z = __fdiv_rn(acc[2], fn);
    o0.w = __fdiv_rn(acc[3], fn);
    o1.x = __fdiv_rn(acc[4], fn);
    o1.y = __fdiv_rn(acc[5], fn);
    o1.z = __fdiv_rn(acc[6], fn);
    o1.w = __fdiv_rn(acc[7], fn);
    reinterpret_cast<float4*>(dst)[2 * part] = o0;
    reinterpret_cast<float4*>(dst)[2 * part + 1] = o1;
}

// ---------------------------------------------------------------------------
// Warp top-K: radix select (4 passes of 8 bits) on order-preserving uint32
// keys of the float scores finds the K-th largest key T; keys > T are all
// selected, keys == T are taken in ascending block order until K.  Output is
// written in ascending block order with ballots.  `s` is in shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ void warp_topk(const float* s, int n, int K, int32_t* __restrict__ out, uint32_t* hist)
{
    const int lane = threadIdx.x & 31;
    uint32_t prefix = 0, pmask = 0;
    int remaining = K;   // how many of the K still to place at or below the current prefix
    for (int shift = 24; shift >= 0; shift -= 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) hist[lane * 8 + i] = 0;
        __syncwarp();
        for (int e = lane; e < n; e += 32) {
            const uint32_t key = order_key(s[e]);
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncwarp();
        // Lane l owns digits [8l, 8l+8).  Count keys with a larger digit.
        uint32_t loc[8];
        uint32_t lsum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            loc[i] = hist[lane * 8 + i];
            lsum += loc[i];
        }
        // suffix sum over lanes (higher lanes own larger digits)
        uint32_t sfx = lsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, sfx, o);
            if (lane + o < 32) sfx += v;
        }
        const uint32_t above = sfx - lsum;   // keys with digit in lanes > lane
        // the digit holding the remaining-th largest lies in the lane with
        // above < remaining <= above + lsum
        const bool mine = (above < (uint32_t)remaining) && ((uint32_t)remaining <= above + lsum);
        const uint32_t ball = __ballot_sync(0xFFFFFFFFu, mine);
        const int owner = __ffs(ball) - 1;
        uint32_t digit = 0, gt = 0;
        if (lane == owner) {
            uint32_t acc = above;
            for (int i = 7; i >= 0; --i) {
                if ((uint32_t)remaining <= acc + loc[i]) {
                    digit = lane * 8 + i;
                    gt = acc;
                    break;
                }
                acc += loc[i];
            }
        }
        digit = __shfl_sync(0xFFFFFFFFu, digit, owner);
        gt = __shfl_sync(0xFFFFFFFFu, gt, owner);
        remaining -= (int)gt;
        prefix |= digit << shift;
        pmask |= 255u << shift;
        __syncwarp();
    }
    // prefix == T; `remaining` keys equal to T are still needed.
    int pos = 0, eq_taken = 0;
    for (int base = 0; base < n; base += 32) {
        const int e = base + lane;
        const uint32_t key = e < n ? order_key(s[e]) : 0u;
        const bool gt = e < n && key > prefix;
        const bool eq = e < n && key == prefix;
        const uint32_t eqb = __ballot_sync(0xFFFFFFFFu, eq);
        const int eq_rank = eq_taken + __popc(eqb & ((1u << lane) - 1u));
        const bool sel = gt || (eq && eq_rank < remaining);
        const uint32_t selb = __ballot_sync(0xFFFFFFFFu, sel);
        if (sel) out[pos + __popc(selb & ((1u << lane) - 1u))] = e;
        pos += __popc(selb);
        eq_taken += __popc(eqb);
    }
}

// ---------------------------------------------------------------------------
// Scores (+ optional selection) for a group of QG query blocks of one head.
// Pooled keys are staged in shared memory in chunks of 128 rows with a row
// pitch of D+1 floats (conflict-free column reads).
// ---------------------------------------------------------------------------
constexpr int QG = 8;
constexpr int KCH = 128;

template <int D>
struct ScoreSmem {
    static constexpr int KP = KCH * (D + 1);   // floats
    static constexpr int QP = QG * D;          // floats
    static constexpr int S = QG * HF_MAX_KEY_BLOCKS;
    static constexpr int HIST = 8 * 256;       // uint32, one histogram per warp
    static constexpr size_t bytes = sizeof(float) * (KP + QP + S) + sizeof(uint32_t) * HIST;
};

template <int D, bool WRITE_SCORES, bool SELECT>
__global__ void __launch_bounds__(256) score_select_kernel(const float* __restrict__ qp, const float* __restrict__ kp,
                                                           Geom g, float* __restrict__ scores,
                                                           int32_t* __restrict__ idx)
{
    extern __shared__ __align__(16) float smf[];
    float* kps = smf;
    float* qps = kps + ScoreSmem<D>::KP;
    float* ss = qps + ScoreSmem<D>::QP;
    uint32_t* hist = reinterpret_cast<uint32_t*>(ss + ScoreSmem<D>::S);

    const int groups = (g.nqb + QG - 1) / QG;
    const int bh = blockIdx.x / groups;
    const int qb0 = (blockIdx.x - bh * groups) * QG;
    const int nq = min(QG, g.nqb - qb0);
    const int tid = threadIdx.x;

    for (int i = tid; i < QG * D; i += 256) {
        const int q = i / D;
        qps[i] = q < nq ? qp[((size_t)bh * g.nqb + qb0 + q) * D + (i - q * D)] : 0.0f;
    }
    const float* kph = kp + (size_t)bh * g.nkb * D;
    for (int base = 0; base < g.nkb; base += KCH) {
        const int rows = min(KCH, g.nkb - base);
        __syncthreads();
        for (int i = tid; i < rows * D; i += 256) {
            const int r = i / D;
            kps[r * (D + 1) + (i - r * D)] = kph[(size_t)base * D + i];
        }
        __syncthreads();
        const int r = tid % KCH;
        const int qh = tid / KCH;   // 0 or 1: query rows qh*4 .. qh*4+3
        if (r < rows) {
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const float* krow = kps + r * (D + 1);
            const float* q0 = qps + (qh * 4) * D;
#pragma unroll 4
            for (int c = 0; c < D; ++c) {
                const float kv = krow[c];
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = __fmaf_rn(q0[i * D + c], kv, acc[i]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) ss[(qh * 4 + i) * HF_MAX_KEY_BLOCKS + base + r] = acc[i] + 0.0f;
        }
    }
    __syncthreads();
    if (WRITE_SCORES) {
        for (int q = 0; q < nq; ++q)
            for (int kb = tid; kb < g.nkb; kb += 256)
                scores[((size_t)bh * g.nqb + qb0 + q) * g.nkb + kb] = ss[q * HF_MAX_KEY_BLOCKS + kb];
    }
    if (SELECT) {
        const int warp = tid / 32;
        if (warp < nq)
            warp_topk(ss + warp * HF_MAX_KEY_BLOCKS, g.nkb, g.k_eff,
                      idx + ((size_t)bh * g.nqb + qb0 + warp) * g.k_eff, hist + warp * 256);
    }
}

// Selection only, from scores in global memory: one warp per row.
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ scores, Geom g,
                                                   int32_t* __restrict__ idx)
{
    extern __shared__ __align__(16) float smf[];
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const long row = (long)blockIdx.x * 8 + warp;
    const long rows = (long)g.BH * g.nqb;
    float* s = smf + warp * HF_MAX_KEY_BLOCKS;
    uint32_t* hist = reinterpret_cast<uint32_t*>(smf + 8 * HF_MAX_KEY_BLOCKS) + warp * 256;
    if (row >= rows) return;
    for (int e = lane; e < g.nkb; e += 32) s[e] = scores[row * g.nkb + e] + 0.0f;
    __syncwarp();
    warp_topk(s, g.nkb, g.k_eff, idx + row * g.k_eff, hist);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes)
{
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

int launch_pool(const uint16_t* Q, const uint16_t* Kc, const Geom& g, const SlotMap& sm, float* qp, float* kp,
                void* stream)
{
    const long tasks = (long)g.BH * (g.nqb + g.nkb);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (g.d == 128) {
        const long grid = (tasks + 15) / 16;
        pool_kernel<128><<<(unsigned)grid, 256, 0, st>>>(Q, Kc, g, sm, qp, kp);
    } else {
        const long grid = (tasks + 31) / 32;
        pool_kernel<64><<<(unsigned)grid, 256, 0, st>>>(Q, Kc, g, sm, qp, kp);
    }
    return (int)cudaGetLastError();
}

template <int D, bool W, bool S>
static int launch_score_t(const float* qp, const float* kp, const Geom& g, float* scores, int32_t* idx,
                          cudaStream_t st)
{
    auto k = score_select_kernel<D, W, S>;
    cudaError_t e = set_smem(k, ScoreSmem<D>::bytes);
    if (e != cudaSuccess) return (int)e;
    const int groups = (g.nqb + QG - 1) / QG;
    k<<<g.BH * groups, 256, ScoreSmem<D>::bytes, st>>>(qp, kp, g, scores, idx);
    return (int)cudaGetLastError();
}

int launch_score_select(const float* qp, const float* kp, const Geom& g, float* scores, int32_t* idx,
                        void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool w = scores != nullptr, s = idx != nullptr;
    if (g.d == 128) {
        if (w && s) return launch_score_t<128, true, true>(qp, kp, g, scores, idx, st);
        if (w) return launch_score_t<128, true, false>(qp, kp, g, scores, idx, st);
        return launch_score_t<128, false, true>(qp, kp, g, scores, idx, st);
    }
    if (w && s) return launch_score_t<64, true, true>(qp, kp, g, scores, idx, st);
    if (w) return launch_score_t<64, true, false>(qp, kp, g, scores, idx, st);
    return launch_score_t<64, false, true>(qp, kp, g, scores, idx, st);
}

int launch_topk(const float* scores, const Geom& g, int32_t* idx, void* stream)
{
    const size_t bytes = sizeof(float) * 8 * HF_MAX_KEY_BLOCKS + sizeof(uint32_t) * 8 * 256;
    cudaError_t e = set_smem(topk_kernel, bytes);
    if (e != cudaSuccess) return (int)e;
    const long rows = (long)g.BH * g.nqb;
    topk_kernel<<<(unsigned)((rows + 7) / 8), 256, bytes, static_cast<cudaStream_t>(stream)>>>(scores, g, idx);
    return (int)cudaGetLastError();
}

}  // namespace hf
