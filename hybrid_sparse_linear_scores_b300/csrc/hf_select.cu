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
// of K (frames of the ring named by `frames`).  D/8 threads per task, each
// owning 8 channels: a thread copies its 16-byte slice of every row of the
// block into shared memory with cp.async (all rows in flight at once, one
// memory round trip), then adds them in token order (sequential float32
// sums).  No data is shared between threads, so no barrier is needed.
// Outputs: qp [BH][nqb][D] (row-major); key pools go to the per-slot cache
// kpc [BH][W slots][D][bpf] (channel-major inside a slot, so that the score
// kernel reads one block's channels with one thread per block).
// ---------------------------------------------------------------------------
constexpr int kPoolThreads = 64;

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gsrc)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

template <int D>
__global__ void __launch_bounds__(kPoolThreads) pool_kernel(const uint16_t* __restrict__ Q,
                                                            const uint16_t* __restrict__ Kc, Geom g, PoolFrames pf,
                                                            float* __restrict__ qp, float* __restrict__ kpc)
{
    constexpr int TPB = D / 8;
    constexpr int TASKS = kPoolThreads / TPB;
    constexpr int ROW = D / 8;   // uint4 per token row
    extern __shared__ __align__(16) uint4 stage[];   // [beta rows][kPoolThreads]
    const int64_t task = (int64_t)blockIdx.x * TASKS + threadIdx.x / TPB;
    const int part = threadIdx.x % TPB;
    const int nq = pf.with_q ? g.nqb : 0;
    const int per_head = nq + pf.n * g.bpf;
    if (task >= (int64_t)g.BH * per_head) return;
    const int bh = (int)(task / per_head);
    const int b = (int)(task - (int64_t)bh * per_head);

    const uint16_t* src;
    int j;
    bool is_q;
    int slot = 0;
    if (b < nq) {
        const int c = b / g.bpf;
        j = b - c * g.bpf;
        src = Q + ((size_t)bh * g.C * g.nf + (size_t)c * g.nf + (size_t)j * g.beta) * D;
        is_q = true;
    } else {
        const int f = (b - nq) / g.bpf;
        j = (b - nq) - f * g.bpf;
        slot = pf.slot[f];
        src = Kc + (((size_t)bh * g.W + slot) * g.slot_stride + (size_t)j * g.beta) * D;
        is_q = false;
    }
    const int n = min(g.beta, g.nf - j * g.beta);
    const uint4* p = reinterpret_cast<const uint4*>(src) + part;
    for (int r = 0; r < n; ++r) cp_async16(&stage[r * kPoolThreads + threadIdx.x], p + (size_t)r * ROW);
    cp_async_wait_all();

    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int r = 0; r < n; ++r) {
        const uint4 v = stage[r * kPoolThreads + threadIdx.x];
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] = __fadd_rn(acc[2 * i], __uint_as_float(w4[i] << 16));
            acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __uint_as_float(w4[i] & 0xFFFF0000u));
        }
    }
    const float fn = static_cast<float>(n);
    if (is_q) {
        float* dst = qp + ((size_t)bh * g.nqb + b) * D + 8 * part;
        reinterpret_cast<float4*>(dst)[0] =
            make_float4(__fdiv_rn(acc[0], fn), __fdiv_rn(acc[1], fn), __fdiv_rn(acc[2], fn), __fdiv_rn(acc[3], fn));
        reinterpret_cast<float4*>(dst)[1] =
            make_float4(__fdiv_rn(acc[4], fn), __fdiv_rn(acc[5], fn), __fdiv_rn(acc[6], fn), __fdiv_rn(acc[7], fn));
    } else {
        float* dst = kpc + (((size_t)bh * g.W + slot) * D + 8 * part) * g.bpf + j;
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[(size_t)i * g.bpf] = __fdiv_rn(acc[i], fn);
    }
}

// ---------------------------------------------------------------------------
// Warp top-K.  Scores are mapped to order-preserving uint32 keys (in place
// over `s`).  The K-th largest key T is found bit by bit from the top: T is
// the largest value with at least K keys >= T (32 warp-wide counts).  Keys
// > T are all selected, keys == T are taken in ascending block order until
// K.  The winners are written in ascending block order with ballots.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ void warp_topk(float* s, int n, int K, int32_t* __restrict__ out)
{
    const int lane = threadIdx.x & 31;
    uint32_t* keys = reinterpret_cast<uint32_t*>(s);
    for (int e = lane; e < n; e += 32) keys[e] = order_key(s[e]);
    __syncwarp();
    uint32_t T = 0;
    if (n <= 256) {   // up to 8 keys per lane, kept in registers
        uint32_t kr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) kr[i] = lane + 32 * i < n ? keys[lane + 32 * i] : 0u;
        const int nmine = n > lane ? (n - lane + 31) / 32 : 0;
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t cand = T | (1u << bit);
            int cnt = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) cnt += (i < nmine && kr[i] >= cand) ? 1 : 0;
            cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
            if (cnt >= K) T = cand;
        }
    } else {
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t cand = T | (1u << bit);
            int cnt = 0;
            for (int e = lane; e < n; e += 32) cnt += keys[e] >= cand ? 1 : 0;
            cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
            if (cnt >= K) T = cand;
        }
    }
    // keys > T: all selected; keys == T: the first (K - #greater) in block order
    int gt_total = 0;
    for (int e = lane; e < n; e += 32) gt_total += keys[e] > T ? 1 : 0;
    gt_total = __reduce_add_sync(0xFFFFFFFFu, gt_total);
    const int remaining = K - gt_total;
    int pos = 0, eq_taken = 0;
    for (int base = 0; base < n; base += 32) {
        const int e = base + lane;
        const uint32_t key = e < n ? keys[e] : 0u;
        const bool gt = e < n && key > T;
        const bool eq = e < n && key == T;
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
// One thread per key block: it copies the block's D pooled channels from the
// slot cache into its own column of shared memory (cp.async, all in flight),
// then runs the QG dot products as separate fixed-order fma chains with the
// query pools broadcast from shared memory.  One warp per query block then
// selects its top K.
// ---------------------------------------------------------------------------
constexpr int QG = 8;

template <int D>
struct ScoreSmem {
    static constexpr int QP = QG * D;          // floats
    static constexpr int S = QG * HF_MAX_KEY_BLOCKS;
    static constexpr int KS = D * 256;         // [D][256]: the key blocks of one pass, one column per thread
    static constexpr size_t bytes = sizeof(float) * (QP + S + KS);
};

template <int D, bool WRITE_SCORES, bool SELECT>
__global__ void __launch_bounds__(256) score_select_kernel(const float* __restrict__ qp, const float* __restrict__ kpc,
                                                           Geom g, SlotMap sm, float* __restrict__ scores,
                                                           int32_t* __restrict__ idx, int32_t* __restrict__ pair_rounds,
                                                           uint32_t* __restrict__ counters)
{
    extern __shared__ __align__(16) float smf[];
    float* qps = smf;
    float* ss = qps + ScoreSmem<D>::QP;
    float* ks = ss + ScoreSmem<D>::S;

    const int groups = (g.nqb + QG - 1) / QG;
    const int bh = blockIdx.x / groups;
    const int qb0 = (blockIdx.x - bh * groups) * QG;
    const int nq = min(QG, g.nqb - qb0);
    const int tid = threadIdx.x;

    for (int i = tid; i < QG * D / 4; i += 256) {
        const int q = (4 * i) / D;
        reinterpret_cast<float4*>(qps)[i] =
            q < nq ? reinterpret_cast<const float4*>(qp + ((size_t)bh * g.nqb + qb0) * D)[i] : make_float4(0, 0, 0, 0);
    }
    __syncthreads();
    for (int kb = tid; kb < g.nkb; kb += 256) {
        const int w = kb / g.bpf;
        const int j = kb - w * g.bpf;
        const float* kcol = kpc + ((size_t)bh * g.W + sm.s[w]) * D * g.bpf + j;
        // this thread's column of the staging area: all D loads in flight at once
#pragma unroll 16
        for (int c = 0; c < D; ++c)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(
                             __cvta_generic_to_shared(ks + c * 256 + tid))),
                         "l"(kcol + (size_t)c * g.bpf)
                         : "memory");
        cp_async_wait_all();
        float acc[QG];
#pragma unroll
        for (int q = 0; q < QG; ++q) acc[q] = 0.0f;
#pragma unroll 4
        for (int c = 0; c < D; c += 4) {
            const float k0 = ks[c * 256 + tid], k1 = ks[(c + 1) * 256 + tid];
            const float k2 = ks[(c + 2) * 256 + tid], k3 = ks[(c + 3) * 256 + tid];
#pragma unroll
            for (int q = 0; q < QG; ++q) {
                const float4 q4 = *reinterpret_cast<const float4*>(qps + q * D + c);
                acc[q] = __fmaf_rn(q4.x, k0, acc[q]);
                acc[q] = __fmaf_rn(q4.y, k1, acc[q]);
                acc[q] = __fmaf_rn(q4.z, k2, acc[q]);
                acc[q] = __fmaf_rn(q4.w, k3, acc[q]);
            }
        }
#pragma unroll
        for (int q = 0; q < QG; ++q) ss[q * HF_MAX_KEY_BLOCKS + kb] = acc[q] + 0.0f;
    }
    __syncthreads();
    if (WRITE_SCORES) {
        for (int q = 0; q < nq; ++q)
            for (int kb = tid; kb < g.nkb; kb += 256)
                scores[((size_t)bh * g.nqb + qb0 + q) * g.nkb + kb] = ss[q * HF_MAX_KEY_BLOCKS + kb];
        if (SELECT) __syncthreads();   // the selection overwrites the rows with keys
    }
    if (SELECT) {
        const int warp = tid / 32;
        if (warp < nq)
            warp_topk(ss + warp * HF_MAX_KEY_BLOCKS, g.nkb, g.k_eff, idx + ((size_t)bh * g.nqb + qb0 + warp) * g.k_eff);
    }
    if (SELECT && pair_rounds) {
        // Rounds of the attention kernel's slab stream for the pairs of tiles this
        // CTA's query blocks form (a pair = 2 tiles of 128 rows = 256/beta query
        // blocks, so QG = 8 blocks hold whole pairs): ceil(#slabs in the union of
        // the pair's selections / 2), with slab k of a frame = rows [64k, 64k+64).
        const int qpp = 256 / g.beta;               // query blocks per pair
        const int npairs = (QG + qpp - 1) / qpp;
        const int spf = (g.nf + 63) / 64;
        const int nsl = g.n_win * spf;
        const int words = (nsl + 31) / 32;
        uint32_t* bits = reinterpret_cast<uint32_t*>(ks);   // [npairs][words], over the staging area
        __syncthreads();                                     // selections written; staging area free
        for (int i = tid; i < npairs * words; i += 256) bits[i] = 0u;
        __syncthreads();
        for (int i = tid; i < nq * g.k_eff; i += 256) {
            const int q = i / g.k_eff;
            const int kb = idx[((size_t)bh * g.nqb + qb0 + q) * g.k_eff + (i - q * g.k_eff)];
            const int w = kb / g.bpf, j = kb - w * g.bpf;
            uint32_t* pb = bits + (q / qpp) * words;
            int s0, s1 = -1;
            if (g.beta == 64) {
                s0 = w * spf + j;
            } else if (g.beta == 128) {
                s0 = w * spf + 2 * j;
                if (2 * j + 1 < spf) s1 = s0 + 1;
            } else {
                s0 = w * spf + (j >> 1);
            }
            atomicOr(&pb[s0 >> 5], 1u << (s0 & 31));
            if (s1 >= 0) atomicOr(&pb[s1 >> 5], 1u << (s1 & 31));
        }
        __syncthreads();
        const int tiles = (g.nqb + 128 / g.beta - 1) / (128 / g.beta);
        const int pairs_per_head = (tiles + 1) / 2;
        const int warp = tid / 32, lane = tid & 31;
        const int pair0 = qb0 / qpp;
        if (warp < npairs && pair0 + warp < pairs_per_head && warp * qpp < nq) {
            int cnt = 0;
            for (int i = lane; i < words; i += 32) cnt += __popc(bits[warp * words + i]);
            cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
            if (lane == 0) {
                const size_t pair = (size_t)bh * pairs_per_head + pair0 + warp;
                pair_rounds[pair] = (cnt + 1) / 2;
                // the attention kernel that follows counts the parts of a split pair
                // here; a launch that gave up part-way can leave a count behind
                counters[2 * pair] = 0u;
                counters[2 * pair + 1] = 0u;
            }
        }
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
    if (row >= rows) return;
    for (int e = lane; e < g.nkb; e += 32) s[e] = scores[row * g.nkb + e] + 0.0f;
    __syncwarp();
    warp_topk(s, g.nkb, g.k_eff, idx + row * g.k_eff);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes)
{
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

int launch_pool(const uint16_t* Q, const uint16_t* Kc, const Geom& g, const PoolFrames& pf, float* qp, float* kpc,
                void* stream)
{
    const long tasks = (long)g.BH * ((pf.with_q ? g.nqb : 0) + pf.n * g.bpf);
    if (tasks == 0) return 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t smem = (size_t)g.beta * kPoolThreads * 16;   // one 16-byte slice per row and thread
    if (g.d == 128) {
        cudaError_t e = set_smem(pool_kernel<128>, smem);
        if (e != cudaSuccess) return (int)e;
        const long grid = (tasks + kPoolThreads / 16 - 1) / (kPoolThreads / 16);
        pool_kernel<128><<<(unsigned)grid, kPoolThreads, smem, st>>>(Q, Kc, g, pf, qp, kpc);
    } else {
        cudaError_t e = set_smem(pool_kernel<64>, smem);
        if (e != cudaSuccess) return (int)e;
        const long grid = (tasks + kPoolThreads / 8 - 1) / (kPoolThreads / 8);
        pool_kernel<64><<<(unsigned)grid, kPoolThreads, smem, st>>>(Q, Kc, g, pf, qp, kpc);
    }
    return (int)cudaGetLastError();
}

template <int D, bool W, bool S>
static int launch_score_t(const float* qp, const float* kpc, const Geom& g, const SlotMap& sm, float* scores,
                          int32_t* idx, int32_t* pair_rounds, uint32_t* counters, cudaStream_t st)
{
    auto k = score_select_kernel<D, W, S>;
    cudaError_t e = set_smem(k, ScoreSmem<D>::bytes);
    if (e != cudaSuccess) return (int)e;
    const int groups = (g.nqb + QG - 1) / QG;
    k<<<g.BH * groups, 256, ScoreSmem<D>::bytes, st>>>(qp, kpc, g, sm, scores, idx, pair_rounds, counters);
    return (int)cudaGetLastError();
}

int launch_score_select(const float* qp, const float* kpc, const Geom& g, const SlotMap& sm, float* scores,
                        int32_t* idx, int32_t* pair_rounds, uint32_t* counters, void* stream)
{
    if (pair_rounds && !counters) return (int)cudaErrorInvalidValue;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool w = scores != nullptr, s = idx != nullptr;
    if (g.d == 128) {
        if (w && s) return launch_score_t<128, true, true>(qp, kpc, g, sm, scores, idx, pair_rounds, counters, st);
        if (w) return launch_score_t<128, true, false>(qp, kpc, g, sm, scores, idx, nullptr, nullptr, st);
        return launch_score_t<128, false, true>(qp, kpc, g, sm, scores, idx, pair_rounds, counters, st);
    }
    if (w && s) return launch_score_t<64, true, true>(qp, kpc, g, sm, scores, idx, pair_rounds, counters, st);
    if (w) return launch_score_t<64, true, false>(qp, kpc, g, sm, scores, idx, nullptr, nullptr, st);
    return launch_score_t<64, false, true>(qp, kpc, g, sm, scores, idx, pair_rounds, counters, st);
}

int launch_topk(const float* scores, const Geom& g, int32_t* idx, void* stream)
{
    const size_t bytes = sizeof(float) * 8 * HF_MAX_KEY_BLOCKS;
    cudaError_t e = set_smem(topk_kernel, bytes);
    if (e != cudaSuccess) return (int)e;
    const long rows = (long)g.BH * g.nqb;
    topk_kernel<<<(unsigned)((rows + 7) / 8), 256, bytes, static_cast<cudaStream_t>(stream)>>>(scores, g, idx);
    return (int)cudaGetLastError();
}

}  // namespace hf
