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
// The kernels are HBM- or latency-bound; none touches tensor cores.  The
// hybrid forward uses fwd_prologue_kernel (query pooling, state operand,
// scores, top-K and the attention kernel's balancing input in one launch) and
// pool_keys_kernel (the pooled-key cache); pool_kernel, score_kernel and
// topk_kernel serve the standalone entry points.
#include <cuda_runtime.h>

#include <cstdint>

#include "hf_internal.h"
#include "hf_ptx.cuh"

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
// kpc [BH][W slots][D/4][bpf][4] (see kp_index).
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

// Pooled-key cache layout inside one ring slot: [D/4][bpf][4] floats (channel
// quads interleaved by block), so that one 16-byte load gives a block four
// consecutive channels and the threads of a warp, one key block each, read
// consecutive 16-byte words.
__device__ __forceinline__ size_t kp_index(int c, int j, int bpf)
{
    return ((size_t)(c >> 2) * bpf + j) * 4 + (c & 3);
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
        float* dst = kpc + ((size_t)bh * g.W + slot) * D * g.bpf;
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[kp_index(8 * part + i, j, g.bpf)] = __fdiv_rn(acc[i], fn);
    }
}

// ---------------------------------------------------------------------------
// Warp top-K.  Scores are mapped to order-preserving uint32 keys (in place
// over `s`).  The K-th largest key T: for up to 256 keys by a bitonic sort in
// registers, beyond that bit by bit from the top (T is the largest value with
// at least K keys >= T; warp-wide counts from ballots, one per 32 keys).
// Keys > T are all selected, keys == T are taken in ascending block order
// until K.
// The winners are written in ascending block order with ballots; on_select(e)
// is called for every winner e.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <typename OnSelect>
__device__ void select_above(const uint32_t* keys, int n, uint32_t T, int remaining, int32_t* __restrict__ out,
                             OnSelect on_select);

// The K-th largest of n <= 256 keys (1 <= K <= n), by one warp: a bitonic
// sort of the keys in registers (8 per lane, element e = 32 r + lane, lanes
// exchanged with shuffles), descending; padding keys are 0, below every key of
// a finite score.  T = element K - 1; the number of keys above T is left to
// the caller.
__device__ __forceinline__ uint32_t warp_kth_largest256(const uint32_t* keys, int n, int K)
{
    const int lane = threadIdx.x & 31;
    uint32_t a[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) a[r] = 32 * r + lane < n ? keys[32 * r + lane] : 0u;
#pragma unroll
    for (int k = 2; k <= 256; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= 32) {   // partner element in this lane's registers
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int p = r ^ (j >> 5);
                    if (p > r) {
                        const bool desc = ((32 * r) & k) == 0;   // k >= 64: the lane bits do not count
                        const uint32_t x = a[r], y = a[p];
                        a[r] = desc ? max(x, y) : min(x, y);
                        a[p] = desc ? min(x, y) : max(x, y);
                    }
                }
            } else {         // partner element in lane ^ j
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, a[r], j);
                    const bool desc = ((32 * r + lane) & k) == 0;
                    const bool lower = (lane & j) == 0;
                    a[r] = (lower == desc) ? max(a[r], y) : min(a[r], y);
                }
            }
        }
    }
    const int rk = (K - 1) >> 5;
    uint32_t v = 0u;
#pragma unroll
    for (int r = 0; r < 8; ++r)
        if (r == rk) v = a[r];
    return __shfl_sync(0xFFFFFFFFu, v, (K - 1) & 31);
}

template <typename OnSelect>
__device__ void warp_topk(float* s, int n, int K, int32_t* __restrict__ out, OnSelect on_select)
{
    const int lane = threadIdx.x & 31;
    uint32_t* keys = reinterpret_cast<uint32_t*>(s);
    for (int e = lane; e < n; e += 32) keys[e] = order_key(s[e]);
    __syncwarp();
    uint32_t T = 0;
    if (n <= 256) {
        T = warp_kth_largest256(keys, n, K);
    } else {   // counts of keys >= c over the warp, bit by bit: one ballot per 32 keys
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t cand = T | (1u << bit);
            int cnt = 0;
            for (int base = 0; base < n; base += 32) {
                const int e = base + lane;
                cnt += __popc(__ballot_sync(0xFFFFFFFFu, e < n && keys[e] >= cand));
            }
            if (cnt >= K) T = cand;
        }
    }
    // keys > T: all selected; keys == T: the first (K - #greater) in block order
    int gt_total = 0;
    for (int base = 0; base < n; base += 32) {
        const int e = base + lane;
        gt_total += __popc(__ballot_sync(0xFFFFFFFFu, e < n && keys[e] > T));
    }
    select_above(keys, n, T, K - gt_total, out, on_select);
}

// The selection itself, once the threshold T is known: every key > T and the
// first `remaining` keys == T in block order, written in ascending block
// order (one warp).
template <typename OnSelect>
__device__ void select_above(const uint32_t* keys, int n, uint32_t T, int remaining, int32_t* __restrict__ out,
                             OnSelect on_select)
{
    const int lane = threadIdx.x & 31;
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
        if (sel) {
            out[pos + __popc(selb & ((1u << lane) - 1u))] = e;
            on_select(e);
        }
        pos += __popc(selb);
        eq_taken += __popc(eqb);
    }
}

__device__ void warp_topk(float* s, int n, int K, int32_t* __restrict__ out)
{
    warp_topk(s, n, K, out, [](int) {});
}

// ---------------------------------------------------------------------------
// Scores for a group of QG query blocks of one head (hf_block_scores).  One
// thread per key block: it copies the block's D pooled channels from the
// slot cache into its own column of shared memory (cp.async, all in flight),
// then runs the QG dot products as separate fixed-order fma chains with the
// query pools broadcast from shared memory.
// ---------------------------------------------------------------------------
constexpr int QG = 8;

template <int D>
struct ScoreSmem {
    static constexpr int QP = QG * D;          // floats
    static constexpr int KS = D * 256;         // [D][256]: the key blocks of one pass, one column per thread
    static constexpr size_t bytes = sizeof(float) * (QP + KS);
};

template <int D>
__global__ void __launch_bounds__(256) score_kernel(const float* __restrict__ qp, const float* __restrict__ kpc,
                                                    Geom g, SlotMap sm, float* __restrict__ scores)
{
    extern __shared__ __align__(16) float smf[];
    float* qps = smf;
    float* ks = qps + ScoreSmem<D>::QP;

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
        const float* kslot = kpc + ((size_t)bh * g.W + sm.s[w]) * D * g.bpf;
        // this thread's column of the staging area: all D loads in flight at once
#pragma unroll 16
        for (int c = 0; c < D; ++c)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(
                             __cvta_generic_to_shared(ks + c * 256 + tid))),
                         "l"(kslot + kp_index(c, j, g.bpf))
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
        for (int q = 0; q < nq; ++q) scores[((size_t)bh * g.nqb + qb0 + q) * g.nkb + kb] = acc[q] + 0.0f;
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

// ---------------------------------------------------------------------------
// Pooling from shared memory.  The rows of up to QG consecutive blocks of one
// frame range are staged as [rows][D] bf16 (one bulk copy); block b covers
// staged rows [r0(b), r0(b) + n(b)).  TPB = NT / QG threads per block, each
// owning CPT consecutive channels, add the block's rows in token order
// (the selection's fixed float32 arithmetic) and divide by the count.
// ---------------------------------------------------------------------------
template <int D, int QG, int NT>
struct PoolLayout {
    static constexpr int TPB = NT / QG;
    static constexpr int CPT = D / TPB >= 1 ? D / TPB : 1;
    static constexpr int ACTIVE = D / CPT;   // threads of a block that own channels
};

template <int CPT>
__device__ __forceinline__ void load_bf16(const uint8_t* p, float (&x)[CPT])
{
    if constexpr (CPT == 1) {
        x[0] = __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(p) << 16);
    } else if constexpr (CPT == 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
        x[0] = bf16_lo(w);
        x[1] = bf16_hi(w);
    } else if constexpr (CPT == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(p);
        x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    } else {
        static_assert(CPT == 8, "channels per thread");
        const uint4 w = *reinterpret_cast<const uint4*>(p);
        x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
        x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
    }
}

// Pools block b (rows [row0, row0 + n) of the staged area) into out[c] for
// this thread's channels; returns false for threads without a block.
template <int D, int QG, int NT>
__device__ __forceinline__ void pool_staged_block(const uint8_t* staged, int b, int nq, int row0, int n,
                                                  float* out /* [D] of block b */)
{
    using L = PoolLayout<D, QG, NT>;
    const int t = threadIdx.x % L::TPB;
    if (b >= nq || t >= L::ACTIVE) return;
    const int c0 = t * L::CPT;
    float acc[L::CPT];
#pragma unroll
    for (int i = 0; i < L::CPT; ++i) acc[i] = 0.0f;
    const uint8_t* src = staged + (size_t)row0 * D * 2 + c0 * 2;
    int r = 0;
    for (; r + 8 <= n; r += 8) {   // eight rows' loads, then their adds in token order
        float x[8][L::CPT];
#pragma unroll
        for (int u = 0; u < 8; ++u) load_bf16<L::CPT>(src + (size_t)(r + u) * D * 2, x[u]);
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int i = 0; i < L::CPT; ++i) acc[i] = __fadd_rn(acc[i], x[u][i]);
    }
    for (; r < n; ++r) {
        float x[L::CPT];
        load_bf16<L::CPT>(src + (size_t)r * D * 2, x);
#pragma unroll
        for (int i = 0; i < L::CPT; ++i) acc[i] = __fadd_rn(acc[i], x[i]);
    }
    const float fn = static_cast<float>(n);
#pragma unroll
    for (int i = 0; i < L::CPT; ++i) out[c0 + i] = __fdiv_rn(acc[i], fn);
}

// One bulk copy of `bytes` (a multiple of 16) from global to shared memory,
// in pieces, completing on `bar` (thread 0 only).
__device__ __forceinline__ void stage_rows(uint8_t* dst, const uint8_t* src, uint32_t bytes, uint64_t* bar)
{
    mbar_arrive_expect_tx(bar, bytes);
    for (uint32_t off = 0; off < bytes; off += 32768u)
        bulk_load(dst + off, src + off, bytes - off < 32768u ? bytes - off : 32768u, bar);
}

// Waits (bounded, every thread) for the staged rows; on a timeout the CTA
// records it and waits once more, bounded, for the copy still in flight.
__device__ __forceinline__ bool wait_staged(uint64_t* bar, const WaitCtl& wc, uint32_t site)
{
    const bool ok = __syncthreads_and(mbar_wait(bar, 0, wc, site) ? 1 : 0) != 0;
    if (!ok && threadIdx.x == 0) {
        const uint32_t a = smem_u32(bar);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(a, 0) && globaltimer_ns() - t0 < wc.limit_ns) {
        }
    }
    return ok;
}

// Shared-memory layout of the two bulk-pooling kernels: up to 256 staged rows,
// reused for the scores once they are pooled.
// Row stride (floats) of the prologue's score rows for nkb key blocks.
__host__ __device__ constexpr int score_stride(int nkb) { return (nkb + 31) & ~31; }

template <int D, int BETA>
struct ProCfg {
    static constexpr int NT = 256;
    static constexpr int QG = 256 / BETA;                      // query blocks of one tile pair
    static constexpr int KB_CH = 32;                           // key-pool channels per staged batch
    static constexpr int STAGE_BYTES = 256 * D * 2;            // query rows, then 2 key-pool batches
    static constexpr int KBUF_BYTES = 2 * KB_CH * NT * 4;
    static constexpr int REGION = STAGE_BYTES > KBUF_BYTES ? STAGE_BYTES : KBUF_BYTES;
    static constexpr int OFF_QP = REGION;                      // fp32 [QG][D]
    static constexpr int OFF_BITS = OFF_QP + QG * D * 4;       // uint32 [2][64]: slabs of tile A / tile B
    static constexpr int OFF_HIST = OFF_BITS + 2 * 64 * 4;     // uint32 [QG][256]: radix-select histograms
    static constexpr int OFF_SEL = OFF_HIST + QG * 256 * 4;    // uint32 [2][QG]: threshold prefix, count above
    static constexpr int OFF_BAR = OFF_SEL + 2 * QG * 4;       // one mbarrier
    static constexpr int OFF_MISC = OFF_BAR + 16;              // uint32 [4]
    static constexpr int OFF_SS = OFF_MISC + 16;               // fp32 [QG][score_stride(nkb)] scores, last:
    static constexpr int SMEM = OFF_SS;                        //   sized per launch by the window's blocks
    static constexpr int SMEM_MAX = OFF_SS + QG * HF_MAX_KEY_BLOCKS * 4;
    // bytes of one launch: the scores of a window of nkb key blocks
    static int smem_for(int nkb) { return OFF_SS + QG * score_stride(nkb) * 4; }
};

// ---------------------------------------------------------------------------
// The hybrid forward's prologue.  CTA = one tile pair of one head (the QG =
// 256 / beta query blocks that the attention kernel processes together):
//   1. one bulk copy of the pair's query rows (contiguous in Q) into shared
//      memory; meanwhile the CTA converts its share of the head's state S
//      into the epilogue's tensor-core operand (bf16 hi = rn(S), lo =
//      rn(S - hi), MN-major, 128-byte swizzle; per head [hi|lo][j/64][c][128 B]);
//   2. pooling of the QG query blocks (fixed float32 arithmetic);
//   3. scores against every key block of the window, from the pooled-key
//      cache (one key block per thread, a fused multiply-add chain in
//      ascending channel order per query block);
//   4. top-K per query block (one warp per block);
//   5. the pair's weight for the attention kernel's balancing: the rounds of
//      its slab stream (slabs: 64 key rows of one frame, in the union of its
//      blocks' selections) in the attention kernel's order, each weighted by
//      round_weight; and its arrival counters zeroed.
// ---------------------------------------------------------------------------
// Weight of a tile pair's slab stream in the attention kernel's order: the
// nI2 = nI & ~1 slabs both tiles need (rounds of both tiles), then
// mp = 2 min(nA / 2, nB / 2) slabs of each tile alone in alternating rounds of
// two, then the rest of tile A's and of tile B's own slabs, then the odd slab
// of both; a round is two consecutive slabs of the stream.
__device__ uint32_t pair_weight(int nI, int nA, int nB)
{
    const int nI2 = nI & ~1, mp = 2 * min(nA >> 1, nB >> 1);
    uint32_t w = (uint32_t)(nI2 / 2) * round_weight(2, 2) +
                 (uint32_t)(mp / 2) * (round_weight(2, 0) + round_weight(0, 2));
    // the rest, A^a B^b I^c, from an even position of the stream
    const int a = nA - mp, c = nI & 1;
    int b = nB - mp;
    w += (uint32_t)(a / 2) * round_weight(2, 0);
    if (a & 1) {   // the last slab of tile A alone shares its round with the next slab
        if (b > 0) {
            w += round_weight(1, 1);
            --b;
        } else {
            return w + (c ? round_weight(2, 1) : round_weight(1, 0));
        }
    }
    w += (uint32_t)(b / 2) * round_weight(0, 2);
    if (b & 1) return w + (c ? round_weight(1, 2) : round_weight(0, 1));
    return w + (c ? round_weight(1, 1) : 0u);
}

template <int D, int BETA>
__global__ void __launch_bounds__(256) fwd_prologue_kernel(const uint16_t* __restrict__ Q,
                                                           const float* __restrict__ kpc,
                                                           const float* __restrict__ S, Geom g, SlotMap sm,
                                                           int32_t* __restrict__ idx, uint16_t* __restrict__ smma,
                                                           int32_t* __restrict__ pair_rounds,
                                                           uint32_t* __restrict__ counters, uint32_t* status,
                                                           uint64_t wait_limit_ns)
{
    using Cfg = ProCfg<D, BETA>;
    constexpr int QG = Cfg::QG;
    extern __shared__ __align__(128) uint8_t smem[];
    float* qps = reinterpret_cast<float*>(smem + Cfg::OFF_QP);
    uint32_t* bits = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_BITS);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);

    const int groups = (g.nqb + QG - 1) / QG;   // tile pairs per head
    const int bh = blockIdx.x / groups;
    const int pair = blockIdx.x - bh * groups;
    const int qb0 = pair * QG;
    const int nq = min(QG, g.nqb - qb0);
    const int tid = threadIdx.x, warp = tid >> 5;
    auto row_of = [&](int qb) { return (qb / g.bpf) * g.nf + (qb % g.bpf) * BETA; };
    auto len_of = [&](int qb) { return min(BETA, g.nf - (qb % g.bpf) * BETA); };
    const int row_start = row_of(qb0);
    const int row_end = row_of(qb0 + nq - 1) + len_of(qb0 + nq - 1);

    if (tid == 0) {
        misc[0] = 0;
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)
        stage_rows(smem, reinterpret_cast<const uint8_t*>(Q + ((size_t)bh * g.C * g.nf + row_start) * D),
                   (uint32_t)(row_end - row_start) * D * 2, bar);

    // 1. this CTA's rows of the state operand, while the query rows arrive
    // (S == nullptr: the workspace already holds the operand of the current S)
    if (S != nullptr) {
        const int rows_per = (D + groups - 1) / groups;
        const int c_lo = min(D, pair * rows_per), c_hi = min(D, c_lo + rows_per);
        uint8_t* base = reinterpret_cast<uint8_t*>(smma) + (size_t)bh * 2 * D * D * 2;
        for (int e = tid; e < (c_hi - c_lo) * (D / 8); e += Cfg::NT) {
            const int c = c_lo + e / (D / 8);
            const int j0 = (e % (D / 8)) * 8;
            const float4* src = reinterpret_cast<const float4*>(S + ((size_t)bh * D + c) * D + j0);
            const float4 a = __ldg(src), b = __ldg(src + 1);
            const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                hi[k] = pack_bf16(x[2 * k], x[2 * k + 1]);
                lo[k] = pack_bf16(x[2 * k] - bf16_lo(hi[k]), x[2 * k + 1] - bf16_hi(hi[k]));
            }
            const uint32_t off = (uint32_t)(j0 / 64) * (uint32_t)(D * 128) + c * 128u +
                                 ((((uint32_t)(j0 % 64) >> 3) ^ ((uint32_t)c & 7u)) << 4);
            *reinterpret_cast<uint4*>(base + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(base + (size_t)D * D * 2 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    }

    // 2. pooling of the pair's query blocks
    const WaitCtl wc{reinterpret_cast<volatile uint32_t*>(misc), status, wait_limit_ns};
    if (!wait_staged(bar, wc, SITE_PROLOGUE_Q)) return;
    {
        const int b = tid / PoolLayout<D, QG, Cfg::NT>::TPB;
        if (b < QG) {
            float* out = qps + b * D;
            if (b < nq)
                pool_staged_block<D, QG, Cfg::NT>(smem, b, nq, row_of(qb0 + b) - row_start, len_of(qb0 + b), out);
            else
                for (int c = tid % PoolLayout<D, QG, Cfg::NT>::TPB; c < D; c += PoolLayout<D, QG, Cfg::NT>::TPB)
                    out[c] = 0.0f;
        }
    }
    __syncthreads();

    // the key pools of the new frames come from the key pooling launched just
    // before this kernel (a programmatic dependency: this kernel may have
    // started while it ran)
    griddep_wait();
    // 3. scores.  A thread's key block: its pooled channels are copied from
    // the cache into the thread's own column of a batch buffer (cp.async,
    // KB_CH channels per batch, two batches over the staged rows, which are no
    // longer needed), the next batch in flight while the fused multiply-add
    // chains run over the current one.
    float* ss = reinterpret_cast<float*>(smem + Cfg::OFF_SS);
    const int sst = score_stride(g.nkb);   // score row stride (floats)
    float4* kbuf = reinterpret_cast<float4*>(smem);   // [2][KB_CH / 4][NT] channel quads
    constexpr int NB = D / Cfg::KB_CH;
    constexpr int NQ4 = Cfg::KB_CH / 4;               // channel quads per batch
    for (int kb0 = 0; kb0 < g.nkb; kb0 += Cfg::NT) {
        const int kb = kb0 + tid;
        const bool have = kb < g.nkb;
        const float* kq = kpc;   // this block's first channel quad in the cache
        if (have) {
            const int w = kb / g.bpf;
            const int j = kb - w * g.bpf;
            kq = kpc + ((size_t)bh * g.W + sm.s[w]) * D * g.bpf + kp_index(0, j, g.bpf);
        }
        auto issue = [&](int b) {
            if (have) {
                float4* dst = kbuf + (b & 1) * NQ4 * Cfg::NT + tid;
#pragma unroll
                for (int u = 0; u < NQ4; ++u)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                                     __cvta_generic_to_shared(dst + u * Cfg::NT))),
                                 "l"(kq + (size_t)(b * NQ4 + u) * g.bpf * 4)
                                 : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        float acc[QG];
#pragma unroll
        for (int q = 0; q < QG; ++q) acc[q] = 0.0f;
        issue(0);
#pragma unroll 1
        for (int b = 0; b < NB; ++b) {
            if (b + 1 < NB) {
                issue(b + 1);
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            } else {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            }
            const float4* kv = kbuf + (b & 1) * NQ4 * Cfg::NT + tid;
#pragma unroll
            for (int u = 0; u < NQ4; ++u) {
                const float4 k4 = kv[u * Cfg::NT];
#pragma unroll
                for (int q = 0; q < QG; ++q) {
                    const float4 qa = *reinterpret_cast<const float4*>(qps + q * D + b * Cfg::KB_CH + 4 * u);
                    acc[q] = __fmaf_rn(qa.x, k4.x, acc[q]);
                    acc[q] = __fmaf_rn(qa.y, k4.y, acc[q]);
                    acc[q] = __fmaf_rn(qa.z, k4.z, acc[q]);
                    acc[q] = __fmaf_rn(qa.w, k4.w, acc[q]);
                }
            }
        }
        if (have) {
#pragma unroll
            for (int q = 0; q < QG; ++q)
                if (q < nq) ss[q * sst + kb] = acc[q] + 0.0f;
        }
    }
    // the pair's slab set (64 key rows of one frame per slab), filled as the
    // blocks are selected
    const int spf = (g.nf + 63) / 64;
    const int words = (g.n_win * spf + 31) / 32;
    for (int i = tid; i < 2 * 64; i += Cfg::NT) bits[i] = 0u;
    __syncthreads();

    // 4. top-K of every query block of the pair.  The K-th largest
    // order-preserving key T of a block: for windows of up to 256 key blocks
    // one warp per query block sorts the block's keys in registers (bitonic);
    // for larger windows a radix select over the whole CTA builds T one byte
    // at a time (all threads histogram the current byte of the keys that
    // match the bytes found so far, shared-memory atomics; then one warp per
    // block finds the byte with a suffix scan).  Then one warp per block
    // writes the keys > T and the first (K - #greater) keys == T in block
    // order, marking their slabs.
    uint32_t* keys = reinterpret_cast<uint32_t*>(ss);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_HIST);
    uint32_t* selP = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_SEL);   // prefix of T
    uint32_t* selG = selP + QG;                                            // keys above the prefix
    const int lane = tid & 31;
    const int nkb = g.nkb, K = g.k_eff;
    for (int i = tid; i < nq * nkb; i += Cfg::NT) {
        const int q = i / nkb, kb = i - q * nkb;
        keys[q * sst + kb] = order_key(ss[q * sst + kb]);
    }
    if (tid < QG) {
        selP[tid] = 0u;
        selG[tid] = 0u;
    }
    // the block of key kb: kb / bpf by a multiply-high (exact for kb, bpf < 2^16)
    const uint32_t bpf_magic = 0xFFFFFFFFu / (uint32_t)g.bpf + 1u;
    // (slab bits per tile: query block q belongs to tile 2 q / QG of the pair)
    auto mark = [&](int kb, int t) {
        uint32_t* bt = bits + 64 * t;
        const int w = (int)__umulhi((uint32_t)kb, bpf_magic), j = kb - w * g.bpf;
        if (BETA == 64) {
            const int s0 = w * spf + j;
            atomicOr(&bt[s0 >> 5], 1u << (s0 & 31));
        } else if (BETA == 128) {
            const int s0 = w * spf + 2 * j;
            atomicOr(&bt[s0 >> 5], 1u << (s0 & 31));
            if (2 * j + 1 < spf) atomicOr(&bt[(s0 + 1) >> 5], 1u << ((s0 + 1) & 31));
        } else {
            const int s0 = w * spf + (j >> 1);
            atomicOr(&bt[s0 >> 5], 1u << (s0 & 31));
        }
    };
    if (nkb <= 256) {
        // one warp per query block: T by a bitonic sort of its keys in registers
        __syncthreads();
        for (int q = warp; q < nq; q += Cfg::NT / 32) {
            const uint32_t* kq = keys + q * sst;
            const uint32_t T = warp_kth_largest256(kq, nkb, K);
            int gt = 0;
            for (int base = 0; base < nkb; base += 32) {
                const int e = base + lane;
                gt += __popc(__ballot_sync(0xFFFFFFFFu, e < nkb && kq[e] > T));
            }
            select_above(kq, nkb, T, K - gt, idx + ((size_t)bh * g.nqb + qb0 + q) * g.k_eff,
                         [&](int kb) { mark(kb, (2 * q) / QG); });
        }
    } else {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < QG * 256; i += Cfg::NT) hist[i] = 0u;
            __syncthreads();
            // (keys of one block crowd into a few bins, most of all at the top
            // byte: lanes with the same bin add once, with their count)
            for (int i0 = 0; i0 < nq * nkb; i0 += Cfg::NT) {
                const int i = i0 + tid;
                int bin = -1;
                if (i < nq * nkb) {
                    const int q = i / nkb, kb = i - q * nkb;
                    const uint32_t k = keys[q * sst + kb];
                    if (shift == 24 || (k >> (shift + 8)) == (selP[q] >> (shift + 8)))
                        bin = q * 256 + (int)((k >> shift) & 255u);
                }
                const uint32_t same = __match_any_sync(0xFFFFFFFFu, bin);
                if (bin >= 0 && lane == __ffs(same) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(same));
            }
            __syncthreads();
            if (warp < nq) {
                const int q = warp;
                uint32_t h[8], local = 0;
                const uint4 h0 = *reinterpret_cast<const uint4*>(hist + q * 256 + 8 * lane);
                const uint4 h1 = *reinterpret_cast<const uint4*>(hist + q * 256 + 8 * lane + 4);
                h[0] = h0.x; h[1] = h0.y; h[2] = h0.z; h[3] = h0.w;
                h[4] = h1.x; h[5] = h1.y; h[6] = h1.z; h[7] = h1.w;
    #pragma unroll
                for (int b = 0; b < 8; ++b) local += h[b];
                uint32_t suff = local;   // keys in the bins of this lane and every higher lane
    #pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, suff, o);
                    if (lane + o < 32) suff += t;
                }
                const uint32_t G = selG[q];
                uint32_t run = G + (suff - local);   // keys above this lane's bins
                int found = -1;
                uint32_t above_found = 0;
    #pragma unroll
                for (int b = 7; b >= 0; --b) {
                    if (found < 0) {
                        if (run + h[b] >= (uint32_t)K) {
                            found = b;
                            above_found = run;
                        }
                        run += h[b];
                    }
                }
                const uint32_t hit = __ballot_sync(0xFFFFFFFFu, found >= 0);
                const int top = 31 - __clz(hit);   // the highest byte value that still keeps K keys
                if (lane == top) {
                    selP[q] |= (uint32_t)(8 * lane + found) << shift;
                    selG[q] = above_found;
                }
            }
            __syncthreads();
        }
        for (int q = warp; q < nq; q += Cfg::NT / 32)
            select_above(keys + q * sst, nkb, selP[q], K - (int)selG[q],
                         idx + ((size_t)bh * g.nqb + qb0 + q) * g.k_eff, [&](int kb) { mark(kb, (2 * q) / QG); });
    }
    if (!pair_rounds) return;

    // 5. the pair's weight: its slabs by tile (both, tile A only, tile B only)
    __syncthreads();
    if (warp == 0) {
        const int lane = tid & 31;
        int nI = 0, nA = 0, nB = 0;
        for (int i = lane; i < words; i += 32) {
            const uint32_t a = bits[i], b = bits[64 + i];
            nI += __popc(a & b);
            nA += __popc(a & ~b);
            nB += __popc(b & ~a);
        }
        nI = __reduce_add_sync(0xFFFFFFFFu, nI);
        nA = __reduce_add_sync(0xFFFFFFFFu, nA);
        nB = __reduce_add_sync(0xFFFFFFFFu, nB);
        if (lane == 0) {
            const size_t pr = (size_t)bh * groups + pair;
            pair_rounds[pr] = (int32_t)pair_weight(nI, nA, nB);
            // the attention kernel that follows counts the parts of a split
            // pair here; a launch that gave up part-way can leave a count behind
            counters[2 * pr] = 0u;
            counters[2 * pr + 1] = 0u;
        }
    }
}

// ---------------------------------------------------------------------------
// Key pooling into the per-slot cache kpc [BH][W slots][D/4][bpf][4].  CTA = one
// key block of one frame of one head (one bulk copy of its rows out of the ring
// slot, 128 threads); the arithmetic is that of the prologue.  Small CTAs, many
// per SM: while some wait for their rows, others pool theirs.
// ---------------------------------------------------------------------------
template <int D, int BETA>
struct KeyPoolCfg {
    static constexpr int NT = 128;
    static constexpr int QG = 1;                        // key blocks per CTA
    static constexpr int STAGE_BYTES = BETA * D * 2;    // the block's rows
    static constexpr int OFF_QP = STAGE_BYTES;          // fp32 [D]: the pooled block
    static constexpr int OFF_BAR = OFF_QP + D * 4;
    static constexpr int OFF_MISC = OFF_BAR + 16;
    static constexpr int SMEM = OFF_MISC + 16;
};

template <int D, int BETA>
__global__ void __launch_bounds__(128) pool_keys_kernel(const uint16_t* __restrict__ Kc, Geom g, PoolFrames pf,
                                                        float* __restrict__ kpc, uint32_t* status,
                                                        uint64_t wait_limit_ns)
{
    using Cfg = KeyPoolCfg<D, BETA>;
    constexpr int QG = Cfg::QG;
    extern __shared__ __align__(128) uint8_t smem[];
    // the forward prologue that follows may start now: it waits for this
    // kernel's pooled keys only before its scores
    griddep_launch_dependents();
    float* qps = reinterpret_cast<float*>(smem + Cfg::OFF_QP);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
    const int gpf = (g.bpf + QG - 1) / QG;   // CTAs per frame
    const int per_head = pf.n * gpf;
    const int bh = blockIdx.x / per_head;
    const int rem = blockIdx.x - bh * per_head;
    const int f = rem / gpf;
    const int j0 = (rem - f * gpf) * QG;
    const int nq = min(QG, g.bpf - j0);
    const int slot = pf.slot[f];
    const int row_start = j0 * BETA;
    const int row_end = min((j0 + nq) * BETA, g.nf);
    const int tid = threadIdx.x;
    if (tid == 0) {
        misc[0] = 0;
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)
        stage_rows(smem,
                   reinterpret_cast<const uint8_t*>(Kc + (((size_t)bh * g.W + slot) * g.slot_stride + row_start) * D),
                   (uint32_t)(row_end - row_start) * D * 2, bar);
    const WaitCtl wc{reinterpret_cast<volatile uint32_t*>(misc), status, wait_limit_ns};
    if (!wait_staged(bar, wc, SITE_POOL_KEYS)) return;
    const int b = tid / PoolLayout<D, QG, Cfg::NT>::TPB;
    if (b < nq)
        pool_staged_block<D, QG, Cfg::NT>(smem, b, nq, b * BETA, min(BETA, g.nf - (j0 + b) * BETA), qps + b * D);
    __syncthreads();
    // qps [QG][D] -> the cache's layout (kp_index): for each channel quad, nq
    // consecutive 16-byte words
    float4* dst = reinterpret_cast<float4*>(kpc + ((size_t)bh * g.W + slot) * D * g.bpf);
    for (int e = tid; e < nq * (D / 4); e += Cfg::NT) {
        const int cq = e / nq, q = e - cq * nq;
        dst[(size_t)cq * g.bpf + j0 + q] = *reinterpret_cast<const float4*>(qps + q * D + 4 * cq);
    }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes)
{
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    // the whole unified L1 as shared memory, so that several CTAs fit per SM
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    return e;
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

template <int D>
static int launch_scores_t(const float* qp, const float* kpc, const Geom& g, const SlotMap& sm, float* scores,
                           cudaStream_t st)
{
    auto k = score_kernel<D>;
    cudaError_t e = set_smem(k, ScoreSmem<D>::bytes);
    if (e != cudaSuccess) return (int)e;
    const int groups = (g.nqb + QG - 1) / QG;
    k<<<g.BH * groups, 256, ScoreSmem<D>::bytes, st>>>(qp, kpc, g, sm, scores);
    return (int)cudaGetLastError();
}

int launch_scores(const float* qp, const float* kpc, const Geom& g, const SlotMap& sm, float* scores, void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return g.d == 128 ? launch_scores_t<128>(qp, kpc, g, sm, scores, st) : launch_scores_t<64>(qp, kpc, g, sm, scores, st);
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

template <int D, int BETA>
static int launch_prologue_t(const uint16_t* Q, const float* kpc, const float* S, const Geom& g, const SlotMap& sm,
                             int32_t* idx, uint16_t* smma, int32_t* pair_rounds, uint32_t* counters,
                             uint32_t* status, uint64_t wait_limit_ns, bool after_pool, cudaStream_t st)
{
    using Cfg = ProCfg<D, BETA>;
    auto k = fwd_prologue_kernel<D, BETA>;
    cudaError_t e = set_smem(k, Cfg::SMEM_MAX);
    if (e != cudaSuccess) return (int)e;
    const int groups = (g.nqb + Cfg::QG - 1) / Cfg::QG;
    // after a key pooling: programmatic stream serialization, the kernel may start
    // while the key pooling runs (it waits for it before its scores).  Otherwise
    // an ordinary launch: whatever ran before may have written Q or S.
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)(g.BH * groups));
    lc.blockDim = dim3(Cfg::NT);
    lc.dynamicSmemBytes = (size_t)Cfg::smem_for(g.nkb);
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = after_pool ? 1 : 0;
    return (int)cudaLaunchKernelEx(&lc, k, Q, kpc, S, g, sm, idx, smma, pair_rounds, counters, status, wait_limit_ns);
}

int launch_fwd_prologue(const uint16_t* Q, const float* kpc, const float* S, const Geom& g, const SlotMap& sm,
                        int32_t* idx, uint16_t* smma, int32_t* pair_rounds, uint32_t* counters, uint32_t* status,
                        uint64_t wait_limit_ns, bool after_pool, void* stream)
{
    if (pair_rounds && !counters) return (int)cudaErrorInvalidValue;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
#define HF_PRO_CASE(DD, BB)                                                                                   \
    if (g.d == DD && g.beta == BB)                                                                            \
        return launch_prologue_t<DD, BB>(Q, kpc, S, g, sm, idx, smma, pair_rounds, counters, status,          \
                                         wait_limit_ns, after_pool, st);
    HF_PRO_CASE(128, 64)
    HF_PRO_CASE(128, 128)
    HF_PRO_CASE(128, 32)
    HF_PRO_CASE(64, 64)
    HF_PRO_CASE(64, 128)
    HF_PRO_CASE(64, 32)
#undef HF_PRO_CASE
    return (int)cudaErrorInvalidValue;
}

template <int D, int BETA>
static int launch_pool_keys_t(const uint16_t* Kc, const Geom& g, const PoolFrames& pf, float* kpc, uint32_t* status,
                              uint64_t wait_limit_ns, cudaStream_t st)
{
    using Cfg = KeyPoolCfg<D, BETA>;
    auto k = pool_keys_kernel<D, BETA>;
    cudaError_t e = set_smem(k, Cfg::SMEM);
    if (e != cudaSuccess) return (int)e;
    const long ctas = (long)g.BH * pf.n * ((g.bpf + Cfg::QG - 1) / Cfg::QG);
    k<<<(unsigned)ctas, Cfg::NT, Cfg::SMEM, st>>>(Kc, g, pf, kpc, status, wait_limit_ns);
    return (int)cudaGetLastError();
}

int launch_pool_keys(const uint16_t* Kc, const Geom& g, const PoolFrames& pf, float* kpc, uint32_t* status,
                     uint64_t wait_limit_ns, void* stream)
{
    if (pf.n == 0) return 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
#define HF_PK_CASE(DD, BB) \
    if (g.d == DD && g.beta == BB) return launch_pool_keys_t<DD, BB>(Kc, g, pf, kpc, status, wait_limit_ns, st);
    HF_PK_CASE(128, 64)
    HF_PK_CASE(128, 128)
    HF_PK_CASE(128, 32)
    HF_PK_CASE(64, 64)
    HF_PK_CASE(64, 128)
    HF_PK_CASE(64, 32)
#undef HF_PK_CASE
    return (int)cudaErrorInvalidValue;
}

}  // namespace hf
