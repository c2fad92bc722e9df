// hf_attn.cu -- block-sparse sliding-window softmax attention on tcgen05,
// with the linear-read + sum epilogue fused in (Hybrid Forcing, English
// technical summary, section 2.A.2 "Block-Sparse Sliding Window Attention"
// and section 2.A.1 "Linear Temporal Attention"; the output is the sum of
// both paths, Spanish technical summary, section 2.A).
//
// Work decomposition.  A tile is 128 query rows = G = 128/beta consecutive
// query blocks of one head; the tensor core's M = 128.  A tile attends to the
// UNION of its blocks' selections, and a row whose own block did not select a
// key block gets -inf logits for it, so every row sees exactly its own
// selection.  Key rows are moved in slabs of 64 rows of one frame (slab k of
// a frame = rows [64k, 64k+64); a slab is one block for beta = 64, half a
// block for beta = 128, two blocks for beta = 32).
//
// The grid is persistent: one CTA per SM, each CTA takes PAIRS of adjacent
// tiles of one head (A and B).  The two tiles share one stream of
// slabs -- the union of both tiles' slabs in window order -- so a slab that
// both need is loaded once.  The stream is cut into rounds of two slabs; a
// tile takes part in a round when it needs one or both of its slabs.  The
// two slabs of a round sit one above the other in shared memory, so when a
// tile needs both, Q K^T is one N = 128 MMA per K step (an N = 64 MMA reads
// as many operand bytes from shared memory per FLOP as it computes, and runs
// at about half the tensor core's rate).
//
// Balancing (fused forward).  Pairs differ in length (their union of
// selections), so whole pairs per CTA leave a long tail.  Instead every CTA
// takes an equal share of all pairs' rounds (the score kernel counts each
// pair's rounds), each pair counted with a few extra units for the fixed cost
// of a part: CTA c runs the rounds in units [cT/G, (c+1)T/G) of the T units
// of the G CTAs, cutting at most two pairs.  Each part of a cut pair leaves its
// (O, m, l) rows in a column-major workspace block; the part that arrives
// last (a per-pair counter) merges all parts in part order -- the result does
// not depend on the order of arrival -- and runs the epilogue.
//
// Warp roles (384 threads = 3 warpgroups, 1 CTA per SM):
//   warps 0-3  build the pair's slab stream (thread 0 issues the Q tiles'
//              loads first: they depend only on the pair); then
//   warp 0     TMA producer of the keys (a ring of NR round stages) and, at
//              the end, of the bf16 hi/lo state S for the fused linear read
//              (into the key ring);
//   warp 2     TMA producer of the values (a second ring of NR round stages).
//              Keys are released as soon as Q K^T has read them, values
//              after P V: each ring runs about NR rounds ahead.
//   warp 1     TMEM owner + MMA issuer (the whole warp runs converged, one
//              elected lane issues: the operands stay warp-uniform and the
//              issue keeps pace with the tensor core), in the order
//                QK_A(0) QK_B(0) | PV_A(r) QK_A(r+1) PV_B(r) QK_B(r+1) | ...
//              so that the tensor core works on one tile while the other
//              tile's softmax runs:
//                S_t  = Q_t K^T          (SS MMA, M=128, N=64 or 128, K=d)
//                O_t += P_t V            (TS MMA, P read from TMEM, N=d)
//                LIN_t = phi(Q_t) S_hi + phi(Q_t) S_lo   (fused epilogue)
//   warps 4-7  softmax of tile A, warps 8-11 softmax of tile B: one TMEM lane
//              (= query row) per thread; online softmax in fp32 (ex2, packed
//              f32x2 arithmetic); the reference max only moves when the
//              running max exceeds it by more than 2^8, and then O is
//              rescaled in TMEM (the tensor core is idle on O_t then: the
//              commit that published S_t covers every earlier P V of the tile);
//              P is written back to TMEM as bf16 over S_t; epilogue
//              O/l + LIN/(phi(q).z + eps) -> bf16 -> TMA store.
// TMEM (512 columns): tile t uses [256t, 256t + d) for O_t and
// [256t + 128, 256t + 256) for S_t / P_t / LIN_t.
//
// Every mbarrier wait is bounded (see hf_ptx.cuh); on expiry the CTA records
// HF_ERR_TIMEOUT in the status word, stops issuing work, drains what it
// issued (bounded) and frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "hf_internal.h"
#include "hf_ptx.cuh"

namespace hf {
namespace {

constexpr int kThreads = 384;
// Registers per thread after the warpgroups re-balance them (setmaxnreg):
// 128 x 64 + 256 x 216 <= 384 x 168, the launch's total (168 per thread is
// the most that 12 warps on 4 sub-partitions can be launched with).
constexpr uint32_t kRegsCtl = 64;
constexpr uint32_t kRegsSoftmax = 216;

__device__ __forceinline__ void bar_all() { asm volatile("bar.sync 0, 384;" ::: "memory"); }
__device__ __forceinline__ void bar_ctl() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Barrier over the whole CTA that also ORs `v` over all threads: every thread
// gets the same answer, whatever is written after the barrier.
__device__ __forceinline__ bool bar_all_or(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 0, 384, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Barrier over one softmax group (128 threads, barrier `id`) that ANDs `v`
// over the group: every thread gets the same answer.
__device__ __forceinline__ bool bar_group_and(uint32_t id, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %2, 0;\n\t"
        "bar.red.and.pred p, %1, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(id), "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

template <uint32_t N>
__device__ __forceinline__ void reg_alloc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <uint32_t N>
__device__ __forceinline__ void reg_dealloc()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <int D, int BETA>
struct AttnCfg {
    static constexpr int TILE_M = 128;
    static constexpr int G = 128 / BETA;                 // query blocks per tile
    static constexpr int SLAB = 64;                      // key rows per slab
    static constexpr int DCH = D / 64;                   // 64-column chunks of a row
    static constexpr int NR = D == 128 ? 2 : 4;          // round stages per ring (K and V)
    static constexpr int Q_BYTES = TILE_M * D * 2;       // one tile
    static constexpr int CHUNK = 2 * SLAB * 128;         // one 64-column chunk of a round stage: 16 KB
    static constexpr int RS_BYTES = DCH * CHUNK;         // one round stage (2 slabs of K, or of V)
    static constexpr int SLAB_BYTES = SLAB * D * 2;
    static constexpr int LIN_BYTES = 2 * D * D * 2;      // S hi + lo (bf16)
    static_assert(LIN_BYTES <= NR * RS_BYTES, "state operands must fit in the key ring");
    static constexpr int MAX_SLABS = 2 * HF_MAX_KEY_BLOCKS;
    static constexpr int OFF_Q = 0;                                   // 2 tiles
    static constexpr int OFF_K = 2 * Q_BYTES;                         // NR round stages
    static constexpr int OFF_V = OFF_K + NR * RS_BYTES;               // NR round stages
    static constexpr int OFF_MASK = OFF_V + NR * RS_BYTES;            // uint32[MAX_SLABS/2]: 16-bit masks
    static constexpr int OFF_LIST = OFF_MASK + MAX_SLABS * 2;         // uint32[MAX_SLABS]
    static constexpr int OFF_CODE = OFF_LIST + MAX_SLABS * 4;         // uint8[MAX_SLABS/2]: round codes
    static constexpr int OFF_BAR = OFF_CODE + MAX_SLABS / 2 + 16;
    static constexpr int NBAR = 32;
    static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;               // uint32[32]
    static constexpr int OFF_Z = OFF_MISC + 128;                      // fp32 [D]: z of the pair's head
    static constexpr int SMEM = OFF_Z + D * 4;
    static constexpr int SMEM_ALLOC = SMEM + 1024;                    // slack for 1 KB alignment
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t IDESC_QK64 = idesc_bf16_f32(128, 64, false, false);
    static constexpr uint32_t IDESC_QK128 = idesc_bf16_f32(128, 128, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, false, true);
    static constexpr uint32_t IDESC_LIN = idesc_bf16_f32(128, D, false, true);
};

// barrier slots
enum {
    B_Q = 0,
    B_IT_FULL = 1,     // 4 (NR): the key stage of round r + 1 and the value stage of r have landed
    B_K_EMPTY = 5,     // 4
    B_V_EMPTY = 13,    // 4 (slots 9..12 unused)
    B_S_FULL = 17,     // 2 (per tile)
    B_P_FULL = 19,     // 2
    B_O_DONE = 21,     // 2
    B_PHIQ = 23,       // 2
    B_LIN_DONE = 25,   // 2
    B_LIN_FULL = 27,
    B_DRAIN = 28,
    B_COUNT = 29
};

// misc words
enum {
    M_TMEM = 0,
    M_ABORT = 1,
    M_NLIST = 2,
    M_CAT = 22,      // 3: slabs needed by both tiles / by tile A only / by tile B only
    M_WCOUNT = 8,    // 4: per-warp counts of the list compaction
    M_PFIRST = 12,   // split mode: the CTA's first pair, and
    M_PREF = 13,     //   the global round at which that pair starts
    M_TOTAL = 14,    //   total rounds of all pairs
    M_FIRSTR = 16,   // 2: first round of the part that each tile takes part in
    M_LASTR = 18,    // 2: last such round (-1: none)
    M_OLD = 20,      // 2: arrival count a tile's part found (split pairs)
    M_SKIPLIN = 26,  // 2: this part does not finish the tile: no linear read
    M_WSUM = 3,      // 4: per-warp weight sums of the list's rounds
    M_RA = 28,       // first round of this part
    M_RB = 29        // end of this part's rounds
};

struct AttnParams {
    Geom g;
    SlotMap sm;
    const int32_t* idx;     // [BH][nqb][k_eff]
    const uint16_t* smma;   // [BH][2][d*d] bf16 MMA-layout state (fused only)
    const float* z;         // [BH][d] (fused only)
    float* o_swa;           // [BH][C*nf][d] (standalone only)
    uint32_t* status;
    uint64_t wait_limit_ns;
    int tiles_per_head;
    int pairs_per_head;
    int total_pairs;
    int spf;                // slabs per frame = ceil(nf / 64)
    // Split mode (all three non-null): every CTA takes an equal share of the
    // rounds of all pairs; a pair cut between CTAs leaves a partial result per
    // part (but the last one to arrive), and the part that arrives last merges them.
    const int32_t* pair_rounds;   // [total_pairs] weight of each pair's slab stream (round_weight units)
    float* partial;               // [grid][2 slots][2 tiles][d + 4 columns][128 rows]: O, m, l
    uint32_t* counters;           // [total_pairs][2] parts arrived per tile; zero between launches
};

// Balancing units: each round of a pair counts round_weight units (its MMA
// work), and each pair counts kPartWeight units ahead of its rounds, so that
// the fixed cost of a part (list build, pipeline fill, epilogue) is shared out
// too.  The prologue writes each pair's total weight; round r of a pair whose
// units start at P starts at unit P + kPartWeight + (weights of rounds < r).
__device__ __forceinline__ uint32_t code_weight(uint32_t code)
{
    return round_weight(__popc(code & 3u), __popc((code >> 2) & 3u));
}

// CTA owning global round x when T rounds are cut into G equal shares
// (CTA c takes rounds [c T / G, (c + 1) T / G)).
// (32-bit division whenever T * (G + 1) fits, as on every workload of a
// realistic size; 64-bit otherwise)
__device__ __forceinline__ int round_owner(uint32_t x, uint32_t T, int G)
{
    if ((uint64_t)T * (uint32_t)(G + 1) < (1ull << 32)) return static_cast<int>(((x + 1) * (uint32_t)G - 1) / T);
    return static_cast<int>((((uint64_t)x + 1) * (uint64_t)G - 1) / T);
}
__device__ __forceinline__ uint32_t share_start(int c, uint32_t T, int G)
{
    if ((uint64_t)T * (uint32_t)(G + 1) < (1ull << 32)) return (uint32_t)c * T / (uint32_t)G;
    return static_cast<uint32_t>((uint64_t)c * T / (uint64_t)G);
}
// With fewer rounds than CTAs some shares are empty; such a CTA takes no part.
__device__ __forceinline__ bool share_nonempty(int c, uint32_t T, int G)
{
    return share_start(c, T, G) < share_start(c + 1, T, G);
}

// Round codes: bit (2t + i) of code[r] is set when tile t needs slab i of
// round r (list position 2r + i).  For one tile, m = (code >> 2t) & 3.
__device__ __forceinline__ uint32_t tile_bits(uint32_t code, int t) { return (code >> (2 * t)) & 3u; }

// Bounded wait for phase `parity` of `bar` without reporting (drains).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns)
{
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(a, parity) && globaltimer_ns() - t0 < limit_ns) {
    }
}

// One ring of round stages (keys or values): loads the slabs of every round
// of the stream, in order, each into the stage of its round.  The issuer's
// iteration i (r = ra - 1 + i, i = 0 .. rb - ra) needs the key stage of round
// r + 1 and the value stage of round r; one barrier per iteration covers both
// (count 2: one arrival per ring, with its bytes), so that the issuer waits
// once per iteration.  The key ring (shift 0) loads round ra + i for
// iteration i, the value ring (shift 1) round ra + i - 1; the iteration with
// no round of a ring gets that ring's arrival without bytes.  Before either
// ring arrives for iteration i >= NR, the issuer has released the key stage
// it used in iteration i - NR (it does so in every iteration but the last):
// the barrier's phase of iteration i - NR has then been waited for, so no
// arrival can land in an earlier phase and the issuer never finds the barrier
// a phase ahead.  Returns the number of iterations the ring arrived on;
// *ok = false if a wait gave up.
template <int D, int BETA>
__device__ __forceinline__ int produce_ring(const CUtensorMap* tm, uint8_t* ring, uint64_t* it_full, uint64_t* empty,
                                            uint64_t* k_empty, const uint32_t* list, int n_list, int ra, int rb,
                                            int bh, int shift, const AttnParams& p, const WaitCtl& wc, uint32_t site,
                                            bool& ok)
{
    using Cfg = AttnCfg<D, BETA>;
    const int n_it = rb - ra + 1;
    int i = 0;
    for (; i < n_it; ++i) {
        const int lr = i - shift;   // round of this ring, counted from ra
        const bool load = lr >= 0 && lr < rb - ra;
        if (i >= Cfg::NR && !mbar_wait(&k_empty[(i - Cfg::NR) % Cfg::NR], ((i - Cfg::NR) / Cfg::NR) & 1, wc, site)) {
            ok = false;
            break;
        }
        if (!load) {
            mbar_arrive(&it_full[i % Cfg::NR]);
            continue;
        }
        const int r = ra + lr;
        const int s = lr % Cfg::NR;
        // the stage's previous round was released (for the key ring: just waited for)
        if (shift != 0 && lr >= Cfg::NR && !mbar_wait(&empty[s], ((lr / Cfg::NR) - 1) & 1, wc, site)) {
            ok = false;
            break;
        }
        const int nq = min(2, n_list - 2 * r);
        uint8_t* st = ring + s * Cfg::RS_BYTES;
        mbar_arrive_expect_tx(&it_full[i % Cfg::NR], nq * Cfg::SLAB_BYTES);
        for (int q = 0; q < nq; ++q) {
            const int slab = static_cast<int>(list[2 * r + q] & 0xFFFFu);
            const int w = slab / p.spf;
            const int k = slab - w * p.spf;
            const int plane = bh * p.g.W + p.sm.s[w];
            for (int m = 0; m < Cfg::DCH; ++m)
                tma_load_3d(st + m * Cfg::CHUNK + q * (Cfg::SLAB * 128), tm, &it_full[i % Cfg::NR], 64 * m, 64 * k,
                            plane);
        }
    }
    return i;
}

template <int D, int BETA, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                const AttnParams p)
{
    using Cfg = AttnCfg<D, BETA>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem + Cfg::OFF_K;
    uint8_t* sV = smem + Cfg::OFF_V;
    uint32_t* sMask = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MASK);
    uint32_t* sList = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_LIST);
    uint8_t* sCode = smem + Cfg::OFF_CODE;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);

    const Geom& g = p.g;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    WaitCtl wc{reinterpret_cast<volatile uint32_t*>(misc + M_ABORT), p.status, p.wait_limit_ns};

    if (tid == 0) misc[M_ABORT] = 0;
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        if (FUSED) prefetch_tmap(&tmO);
    }
    if (warp == 1) {
        tmem_alloc(misc + M_TMEM, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[M_TMEM];

    // ---- split mode: the share of all pairs' rounds this CTA takes ----
    const bool split = p.pair_rounds != nullptr;
    uint32_t T = 0, s_c = 0, e_c = 0;
    if (split) {
        // [kThreads] scratch in the slab list, which only ever sees ordinary loads and
        // stores (TMA never writes it) and is first filled by the first pair's list
        int* tsum = reinterpret_cast<int*>(sList);
        static_assert(Cfg::MAX_SLABS >= kThreads, "the prologue's scratch fits in the slab list");
        const int NP = p.total_pairs;
        const int per = (NP + kThreads - 1) / kThreads;
        const int b0 = min(NP, tid * per), b1 = min(NP, b0 + per);
        int loc = 0;
        for (int i = b0; i < b1; ++i) loc += p.pair_rounds[i] + (int)kPartWeight;
        tsum[tid] = loc;
        if (tid == 0) {
            misc[M_PFIRST] = (uint32_t)NP;   // none, unless found below
            misc[M_PREF] = 0;
        }
        __syncthreads();
        if (warp == 0) {   // exclusive scan of the kThreads chunk sums
            constexpr int PL = kThreads / 32;
            int v[PL], ls = 0;
#pragma unroll
            for (int k = 0; k < PL; ++k) {
                v[k] = tsum[lane * PL + k];
                ls += v[k];
            }
            int inc = ls;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int nb = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= o) inc += nb;
            }
            int ex = inc - ls;
#pragma unroll
            for (int k = 0; k < PL; ++k) {
                tsum[lane * PL + k] = ex;
                ex += v[k];
            }
            if (lane == 31) misc[M_TOTAL] = (uint32_t)inc;
        }
        __syncthreads();
        T = misc[M_TOTAL];
        s_c = share_start(blockIdx.x, T, gridDim.x);
        e_c = share_start(blockIdx.x + 1, T, gridDim.x);
        uint32_t P = (uint32_t)tsum[tid];
        for (int i = b0; i < b1; ++i) {
            const uint32_t R = (uint32_t)p.pair_rounds[i] + kPartWeight;   // units of the pair
            if (P <= s_c && s_c < P + R) {
                misc[M_PFIRST] = (uint32_t)i;
                misc[M_PREF] = P;
            }
            P += R;
        }
        __syncthreads();
    }
    const int pair_first = split ? (int)misc[M_PFIRST] : (int)blockIdx.x;
    const uint32_t pref_first = split ? misc[M_PREF] : 0u;

    // the tiles of pair `pair`: head bh, first query block qb0[t], blocks nblk[t] (0 = no tile B)
    auto pair_geometry = [&](int pair, int& bh, int (&qb0)[2], int (&nblk)[2]) {
        bh = pair / p.pairs_per_head;
        const int pr = pair - bh * p.pairs_per_head;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int tile = 2 * pr + t;
            qb0[t] = tile * Cfg::G;
            nblk[t] = tile < p.tiles_per_head ? min(Cfg::G, g.nqb - qb0[t]) : 0;
        }
    };

    if (warp < 4) {
        // ======== warpgroup 0: slab stream, TMA producers, MMA issuer ========
        reg_dealloc<kRegsCtl>();
        int pair = pair_first;
        uint32_t P = pref_first;
        for (;;) {
            // this part of the pair: the pair's units [lo, hi) (counted from its
            // round 0); its rounds [ra, rb), the rounds that start there, follow from
            // the rounds' weights once the slab list is built
            int ra = 0, rb = 1 << 30;
            uint32_t R = 0, lo = 0, hi = 0xFFFFFFFFu;
            if (split) {
                if (pair >= p.total_pairs || P + kPartWeight >= e_c || s_c >= e_c) break;
                R = (uint32_t)p.pair_rounds[pair];    // the pair's weight
                const uint32_t Pr = P + kPartWeight;   // unit of the pair's round 0
                lo = max(s_c, Pr) - Pr;
                hi = min(e_c, Pr + R) - Pr;
            } else if (pair >= p.total_pairs) {
                break;
            }
            int bh, qb0[2], nblk[2];
            pair_geometry(pair, bh, qb0, nblk);
            // ---- barriers (no asynchronous operation is pending here) ----
            if (tid == 0) {
                mbar_init(&bar[B_Q], 1);
                for (int s = 0; s < Cfg::NR; ++s) {
                    mbar_init(&bar[B_IT_FULL + s], 2);   // one arrival per ring producer
                    mbar_init(&bar[B_K_EMPTY + s], 1);
                    mbar_init(&bar[B_V_EMPTY + s], 1);
                }
                for (int t = 0; t < 2; ++t) {
                    mbar_init(&bar[B_S_FULL + t], 1);
                    mbar_init(&bar[B_P_FULL + t], 4);   // one arrival per softmax warp
                    mbar_init(&bar[B_O_DONE + t], 1);
                    mbar_init(&bar[B_PHIQ + t], 128);
                    mbar_init(&bar[B_LIN_DONE + t], 1);
                }
                mbar_init(&bar[B_LIN_FULL], 1);
                mbar_init(&bar[B_DRAIN], 1);
                misc[M_SKIPLIN] = misc[M_SKIPLIN + 1] = 0u;
                fence_mbar_init();
                // the Q tiles depend only on the pair, so they load while the list is built
                // (the previous pair's output store has finished reading the Q region)
                const int ntiles = (nblk[0] > 0) + (nblk[1] > 0);
                // (with the fused epilogue, z of the head rides along: the
                // linear read's denominators then read it from shared memory)
                mbar_arrive_expect_tx(&bar[B_Q], ntiles * Cfg::G * Cfg::DCH * BETA * 128 + (FUSED ? D * 4 : 0));
                if (FUSED) bulk_load(smem + Cfg::OFF_Z, p.z + (size_t)bh * D, D * 4, &bar[B_Q]);
                for (int t = 0; t < 2; ++t) {
                    if (nblk[t] == 0) continue;
                    uint8_t* sQ = smem + Cfg::OFF_Q + t * Cfg::Q_BYTES;
                    for (int gq = 0; gq < Cfg::G; ++gq) {
                        const int qb = qb0[t] + min(gq, nblk[t] - 1);   // missing blocks: reload the last one
                        const int c = qb / g.bpf;
                        const int j = qb - c * g.bpf;
                        for (int m = 0; m < Cfg::DCH; ++m)
                            tma_load_3d(sQ + m * (Cfg::TILE_M * 128) + gq * BETA * 128, &tmQ, &bar[B_Q], 64 * m,
                                        j * BETA, bh * g.C + c);
                    }
                }
            }
            // ---- the pair's slab stream ----
            // mask bits of slab s: tile t, sub-block h (beta = 32 only), query
            // block gq of the tile -> bit 8t + 4h + gq.
            const int nsl = g.n_win * p.spf;
            for (int i = tid; i < (nsl + 1) / 2; i += 128) sMask[i] = 0;
            bar_ctl();
            {
                // entry i of tile t: query block i / k_eff of the tile, key block kb
                auto mark = [&](int t, int i, int kb) {
                    const int gq = i / g.k_eff;
                    if (kb < 0 || kb >= g.nkb) {
                        report_error(wc, HF_DEV_ERR_CHECK, SITE_ATTN_BAD_INDEX);
                        return;
                    }
                    const int w = kb / g.bpf;
                    const int j = kb - w * g.bpf;
                    if (BETA == 64) {
                        const int s = w * p.spf + j;
                        atomicOr(&sMask[s >> 1], (1u << (8 * t + gq)) << ((s & 1) * 16));
                    } else if (BETA == 128) {
                        const int s = w * p.spf + 2 * j;
                        atomicOr(&sMask[s >> 1], (1u << (8 * t)) << ((s & 1) * 16));
                        if (2 * j + 1 < p.spf)
                            atomicOr(&sMask[(s + 1) >> 1], (1u << (8 * t)) << (((s + 1) & 1) * 16));
                    } else {
                        const int s = w * p.spf + (j >> 1);
                        atomicOr(&sMask[s >> 1], (1u << (8 * t + 4 * (j & 1) + gq)) << ((s & 1) * 16));
                    }
                };
                int total[2];
                const int32_t* ip[2];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    total[t] = nblk[t] * g.k_eff;
                    ip[t] = p.idx + ((size_t)bh * g.nqb + qb0[t]) * g.k_eff;
                }
                // the first 128 entries of both tiles in one memory round trip
                const int kb0 = tid < total[0] ? __ldg(ip[0] + tid) : 0;
                const int kb1 = tid < total[1] ? __ldg(ip[1] + tid) : 0;
                if (tid < total[0]) mark(0, tid, kb0);
                if (tid < total[1]) mark(1, tid, kb1);
#pragma unroll
                for (int t = 0; t < 2; ++t)
                    for (int i = tid + 128; i < total[t]; i += 128) mark(t, i, __ldg(ip[t] + i));
            }
            bar_ctl();
            {   // The slabs that either tile needs, ordered so that the rounds (pairs of
                // consecutive list entries) keep both tiles busy: (1) slabs both tiles
                // need, two per round; (2) rounds of two slabs only tile A needs
                // alternating with rounds of two only tile B needs, so that one tile's
                // softmax runs while the tensor core works on the other tile; (3) the
                // rest of the longer side; (4) the odd slab of (1), if any.  Window
                // order within each group.  The count of rounds is ceil(n / 2) as in
                // any order.
                auto cat_of = [](uint32_t m) -> int {
                    return m == 0u ? 0 : ((m & 0x00FFu) && (m & 0xFF00u)) ? 1 : ((m & 0x00FFu) ? 2 : 3);
                };
                if (tid < 3) misc[M_CAT + tid] = 0;
                bar_ctl();
                {
                    int c1 = 0, c2 = 0, c3 = 0;
                    for (int s = tid; s < nsl; s += 128) {
                        const int c = cat_of((sMask[s >> 1] >> ((s & 1) * 16)) & 0xFFFFu);
                        c1 += c == 1;
                        c2 += c == 2;
                        c3 += c == 3;
                    }
                    c1 = __reduce_add_sync(0xFFFFFFFFu, c1);
                    c2 = __reduce_add_sync(0xFFFFFFFFu, c2);
                    c3 = __reduce_add_sync(0xFFFFFFFFu, c3);
                    if (lane == 0) {
                        atomicAdd(&misc[M_CAT + 0], (uint32_t)c1);
                        atomicAdd(&misc[M_CAT + 1], (uint32_t)c2);
                        atomicAdd(&misc[M_CAT + 2], (uint32_t)c3);
                    }
                }
                bar_ctl();
                const int nI = (int)misc[M_CAT], nA = (int)misc[M_CAT + 1], nB = (int)misc[M_CAT + 2];
                const int base_out = nI + nA + nB;
                const int nI2 = nI & ~1;
                const int mp = 2 * min(nA >> 1, nB >> 1);   // slabs of each side in the alternating part
                int run[3] = {0, 0, 0};                     // slabs of each group placed by earlier chunks
                for (int base = 0; base < nsl; base += 128) {
                    const int s = base + tid;
                    const uint32_t m = s < nsl ? (sMask[s >> 1] >> ((s & 1) * 16)) & 0xFFFFu : 0u;
                    const int cat = cat_of(m);
                    uint32_t ball[3];
#pragma unroll
                    for (int k = 0; k < 3; ++k) ball[k] = __ballot_sync(0xFFFFFFFFu, cat == k + 1);
                    if (lane == 0)
                        misc[M_WCOUNT + warp] = (uint32_t)__popc(ball[0]) | ((uint32_t)__popc(ball[1]) << 8) |
                                                ((uint32_t)__popc(ball[2]) << 16);
                    bar_ctl();
                    int before[3] = {run[0], run[1], run[2]}, tot[3] = {0, 0, 0};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t w = misc[M_WCOUNT + q];
#pragma unroll
                        for (int k = 0; k < 3; ++k) {
                            const int c = (int)((w >> (8 * k)) & 0xFFu);
                            if (q < warp) before[k] += c;
                            tot[k] += c;
                        }
                    }
                    if (cat != 0) {
                        const int k = cat - 1;
                        const int q = before[k] + __popc(ball[k] & ((1u << lane) - 1u));
                        int pos;
                        if (k == 0)
                            pos = q < nI2 ? q : base_out - 1;
                        else if (k == 1)
                            pos = q < mp ? nI2 + 2 * (q & ~1) + (q & 1) : nI2 + mp + q;
                        else
                            pos = q < mp ? nI2 + 2 * (q & ~1) + 2 + (q & 1) : nI2 + nA + q;
                        sList[pos] = static_cast<uint32_t>(s) | (m << 16);
                    }
#pragma unroll
                    for (int k = 0; k < 3; ++k) run[k] += tot[k];
                    bar_ctl();
                }
                if (tid == 0) {
                    misc[M_NLIST] = base_out;
                    misc[M_FIRSTR] = misc[M_FIRSTR + 1] = 0x7FFFFFFFu;
                    misc[M_LASTR] = misc[M_LASTR + 1] = 0xFFFFFFFFu;
                    misc[M_RA] = misc[M_RB] = 0u;
                }
                for (int r = tid; r < (base_out + 1) / 2; r += 128) {
                    uint32_t c = 0;
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        if (2 * r + i < base_out) {
                            const uint32_t e = sList[2 * r + i];
                            if (e & 0x00FF0000u) c |= 1u << i;
                            if (e & 0xFF000000u) c |= 4u << i;
                        }
                    }
                    sCode[r] = static_cast<uint8_t>(c);
                }
                bar_ctl();
                {   // The part's rounds: round r starts at the sum of the weights of the
                    // rounds before it; this part takes the rounds that start in [lo, hi)
                    // (the neighbouring CTA's share starts where this one ends, so every
                    // round has exactly one owner).  Each thread sums a run of
                    // consecutive rounds; a scan over the runs gives every start.
                    const int nr = (base_out + 1) / 2;
                    const int CH = (nr + 127) / 128;
                    const int r0 = min(nr, tid * CH), r1 = min(nr, r0 + CH);
                    uint32_t wsum = 0;
                    for (int r = r0; r < r1; ++r) wsum += code_weight(sCode[r]);
                    uint32_t inc = wsum;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                        if (lane >= o) inc += v;
                    }
                    if (lane == 31) misc[M_WSUM + warp] = inc;
                    bar_ctl();
                    uint32_t st = inc - wsum, total = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t wq = misc[M_WSUM + q];
                        if (q < warp) st += wq;
                        total += wq;
                    }
                    uint32_t n_lo = 0, n_hi = 0;
                    for (int r = r0; r < r1; ++r) {
                        n_lo += st < lo ? 1u : 0u;
                        n_hi += st < hi ? 1u : 0u;
                        st += code_weight(sCode[r]);
                    }
                    n_lo = __reduce_add_sync(0xFFFFFFFFu, n_lo);
                    n_hi = __reduce_add_sync(0xFFFFFFFFu, n_hi);
                    if (lane == 0) {
                        atomicAdd(&misc[M_RA], n_lo);
                        atomicAdd(&misc[M_RB], n_hi);
                    }
                    // the prologue's weight of the pair is the weight of this list
                    if (tid == 0 && split && total != R) report_error(wc, HF_DEV_ERR_CHECK, SITE_ATTN_BAD_INDEX);
                    bar_ctl();
                    ra = (int)misc[M_RA];
                    rb = (int)misc[M_RB];
                }
                // first and last round of this part that each tile takes part in
                const int rend = min(rb, (base_out + 1) / 2);
                for (int r = ra + tid; r < rend; r += 128) {
                    const uint32_t c = sCode[r];
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (tile_bits(c, t)) {
                            atomicMin(reinterpret_cast<int*>(&misc[M_FIRSTR + t]), r);
                            atomicMax(reinterpret_cast<int*>(&misc[M_LASTR + t]), r);
                        }
                    }
                }
            }
            // list and barriers ready; a bad index: nothing more of this pair is issued
            // (the Q load in flight lands first)
            if (bar_all_or(*wc.abort_flag != 0)) {
                if (tid == 0) drain_wait(&bar[B_Q], 0, p.wait_limit_ns);
                break;
            }
            const int n_list = (int)misc[M_NLIST];
            const int n_rounds = (n_list + 1) / 2;
            rb = min(rb, n_rounds);

            if (warp == 0 && lane == 0) {
                // ---------- key ring, state operand (Q was issued at the pair's start) ----------
                bool ok = true;
                const int issued = produce_ring<D, BETA>(&tmK, sK, &bar[B_IT_FULL], &bar[B_K_EMPTY], &bar[B_K_EMPTY],
                                                         sList, n_list, ra, rb, bh, 0, p, wc, SITE_ATTN_KV_EMPTY, ok);
                bool lin_issued = false;
                if (FUSED && ok) {
                    // the state operands go into the key ring once every key stage is free
                    for (int lr = max(0, rb - ra - Cfg::NR); lr < rb - ra && ok; ++lr)
                        ok = mbar_wait(&bar[B_K_EMPTY + lr % Cfg::NR], (lr / Cfg::NR) & 1, wc, SITE_ATTN_KV_EMPTY);
                    if (ok) {
                        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.smma) + (size_t)bh * Cfg::LIN_BYTES;
                        mbar_arrive_expect_tx(&bar[B_LIN_FULL], Cfg::LIN_BYTES);
                        bulk_load(sK, src, Cfg::LIN_BYTES / 2, &bar[B_LIN_FULL]);
                        bulk_load(sK + Cfg::LIN_BYTES / 2, src + Cfg::LIN_BYTES / 2, Cfg::LIN_BYTES / 2,
                                  &bar[B_LIN_FULL]);
                        lin_issued = true;
                    }
                }
                // drain (bounded): every load issued has landed before the pair ends
                for (int i = max(0, issued - Cfg::NR); i < issued; ++i)
                    drain_wait(&bar[B_IT_FULL + i % Cfg::NR], (i / Cfg::NR) & 1, p.wait_limit_ns);
                drain_wait(&bar[B_Q], 0, p.wait_limit_ns);
                if (lin_issued) drain_wait(&bar[B_LIN_FULL], 0, p.wait_limit_ns);
                if (!ok) *wc.abort_flag = 1;
            } else if (warp == 2 && lane == 0) {
                // ---------- value ring ----------
                bool ok = true;
                const int issued = produce_ring<D, BETA>(&tmV, sV, &bar[B_IT_FULL], &bar[B_V_EMPTY], &bar[B_K_EMPTY],
                                                         sList, n_list, ra, rb, bh, 1, p, wc, SITE_ATTN_KV_EMPTY, ok);
                for (int i = max(0, issued - Cfg::NR); i < issued; ++i)
                    drain_wait(&bar[B_IT_FULL + i % Cfg::NR], (i / Cfg::NR) & 1, p.wait_limit_ns);
                if (!ok) *wc.abort_flag = 1;
            } else if (warp == 1) {
                // ---------- MMA issuer (the whole warp, converged; one elected lane issues) ----------
                // Batches in the order A(-1) B(-1) A(0) B(0) A(1) ..., batch t(r) =
                // P V_t(r) followed by Q K^T_t(r+1) (S_t is free again once P V_t(r) has
                // been issued: the tensor core executes in issue order).  Each tile's
                // softmax then runs while the tensor core works on the other tile's
                // batch.
                // waits are polled by every lane and agreed on, so the warp stays converged
                auto wait_all = [&](uint64_t* b, uint32_t parity, uint32_t site) -> bool {
                    return __all_sync(0xFFFFFFFFu, mbar_wait(b, parity, wc, site));
                };
                bool ok = wait_all(&bar[B_Q], 0, SITE_ATTN_Q);
                tc_fence_after();
                // base descriptors (start addresses advance in 16-byte units): Q tiles and
                // the key ring K-major, the value ring MN-major (64-column chunks CHUNK apart)
                const uint64_t q_desc0 = smem_desc(smem_u32(smem + Cfg::OFF_Q), 16, 1024);
                const uint64_t q_desc1 = smem_desc(smem_u32(smem + Cfg::OFF_Q + Cfg::Q_BYTES), 16, 1024);
                const uint64_t k_desc = smem_desc(smem_u32(sK), 16, 1024);
                const uint64_t v_desc = smem_desc(smem_u32(sV), Cfg::CHUNK, 1024);
                // last round of this part each tile takes part in (-1: none)
                const int last_round0 = (int)misc[M_LASTR + 0];
                const int last_round1 = (int)misc[M_LASTR + 1];
                int cnt0 = 0, cnt1 = 0;
                bool first0 = true, first1 = true;
                // One loop body for every batch, so that each batch's code exists once
                // (the issuer then runs from a small stretch of code): for r = ra - 1
                // .. rb - 1 and t = A, B: P V_t(r) (r >= ra), then Q K^T_t(r + 1)
                // (r + 1 < rb).  Round codes are read one round ahead of their use.
                // The tensor core only stays busy while MMAs are issued back to back:
                // any other work of this thread between two MMAs idles it for that time
                // plus a restart.  So the stages of both batches of an iteration are
                // waited for once, before the first P, and the usual batch (both slabs
                // of both rounds) is issued in one block without any other instruction.
                uint32_t c_cur = 0u;
                uint32_t c_nxt = ra < rb ? sCode[ra] : 0u;
#pragma unroll 1
                for (int r = ra - 1; ok && r < rb; ++r) {
                    const bool more = r + 1 < rb;
                    const int sv = (r - ra) % Cfg::NR;       // value stage of r (r >= ra)
                    const int sk = (r + 1 - ra) % Cfg::NR;   // key stage of r + 1
                    {   // the key stage of r + 1 and the value stage of r: one barrier
                        const int it = r + 1 - ra;
                        ok = wait_all(&bar[B_IT_FULL + it % Cfg::NR], (it / Cfg::NR) & 1, SITE_ATTN_KV_FULL);
                    }
#pragma unroll 1
                    for (int t = 0; t < 2 && ok; ++t) {
                        const uint32_t m_pv = r >= ra ? tile_bits(c_cur, t) : 0u;
                        const uint32_t m_qk = more ? tile_bits(c_nxt, t) : 0u;
                        int& cnt = t ? cnt1 : cnt0;
                        bool& first = t ? first1 : first0;
                        const int last_round = t ? last_round1 : last_round0;
                        if (m_pv != 0u) {
                            ok = wait_all(&bar[B_P_FULL + t], cnt & 1, SITE_ATTN_P_FULL);
                            ++cnt;
                            if (!ok) break;
                        }
                        tc_fence_after();
                        const uint32_t o_tm = tmem + 256 * t;
                        const uint64_t qd = t ? q_desc1 : q_desc0;
                        bool done = false;
                        if constexpr (D == 128) {
                            if (m_pv == 3u && m_qk == 3u && r != last_round) {
                                const uint64_t vd0 = v_desc + (uint64_t)((sv * Cfg::RS_BYTES) >> 4);
                                const uint64_t kd = k_desc + (uint64_t)((sk * Cfg::RS_BYTES) >> 4);
                                static_assert(Cfg::SLAB / 16 == 4, "four K steps per slab");
                                mma_attn_batch_warp<(2048 >> 4), (Cfg::CHUNK >> 4)>(
                                    o_tm, o_tm + 128, vd0, vd0 + (uint64_t)((Cfg::SLAB * 128) >> 4), Cfg::IDESC_PV,
                                    first ? 0u : 1u, o_tm + 128, qd, kd, Cfg::IDESC_QK128, &bar[B_V_EMPTY + sv],
                                    &bar[B_S_FULL + t], &bar[B_K_EMPTY + sk], t == 1 ? 1u : 0u);
                                first = false;
                                done = true;
                            }
                        }
                        if (!done) {
                            if (m_pv != 0u) {
                                const int n = m_pv == 3u ? 2 : 1;
#pragma unroll
                                for (int j = 0; j < 2; ++j) {
                                    if (j >= n) break;
                                    const int i = (m_pv == 2u) ? 1 : j;   // slab of the round; P columns [32j, 32j + 32)
                                    const uint64_t vd =
                                        v_desc + (uint64_t)((sv * Cfg::RS_BYTES + i * Cfg::SLAB * 128) >> 4);
                                    static_assert(Cfg::SLAB / 16 == 4, "four K steps per slab");
                                    mma_ts_k4_warp<(2048 >> 4)>(o_tm, o_tm + 128 + 32 * j, vd, Cfg::IDESC_PV,
                                                                (first && j == 0) ? 0u : 1u);
                                }
                                first = false;
                                if (r == last_round) mma_commit_warp(&bar[B_O_DONE + t]);
                            }
                            if (t == 1 && r >= ra) mma_commit_warp(&bar[B_V_EMPTY + sv]);
                            if (m_qk != 0u) {
                                // both slabs: one N = 128 operand; one slab: its 64 rows
                                const uint64_t kd =
                                    k_desc + (uint64_t)((sk * Cfg::RS_BYTES + (m_qk == 2u ? Cfg::SLAB * 128 : 0)) >> 4);
                                const uint32_t idesc = m_qk == 3u ? Cfg::IDESC_QK128 : Cfg::IDESC_QK64;
                                static_assert(D == 64 || Cfg::TILE_M * 128 == Cfg::CHUNK, "one chunk stride for Q and K");
                                mma_ss_kloop_warp<D / 16, (Cfg::CHUNK >> 4)>(o_tm + 128, qd, kd, idesc, 0u);
                                mma_commit_warp(&bar[B_S_FULL + t]);
                            }
                            if (t == 1 && more) mma_commit_warp(&bar[B_K_EMPTY + sk]);
                        }
                    }
                    c_cur = c_nxt;
                    c_nxt = r + 2 < rb ? sCode[r + 2] : 0u;
                }
                if (FUSED && ok) {
                    ok = wait_all(&bar[B_LIN_FULL], 0, SITE_ATTN_LIN);
                    const uint64_t l_desc = smem_desc(smem_u32(sK), D * 128, 1024);
                    for (int t = 0; ok && t < 2; ++t) {
                        if (nblk[t] == 0) continue;
                        ok = wait_all(&bar[B_PHIQ + t], 0, SITE_ATTN_PHIQ);
                        if (!ok) break;
                        if (*reinterpret_cast<volatile uint32_t*>(&misc[M_SKIPLIN + t]) != 0u) continue;
                        tc_fence_after();
                        const uint64_t qd = t ? q_desc1 : q_desc0;
#pragma unroll
                        for (int hl = 0; hl < 2; ++hl) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_ss_warp(tmem + 256 * t + 128,
                                       qd + (uint64_t)(((kk >> 2) * (Cfg::TILE_M * 128) + (kk & 3) * 32) >> 4),
                                       l_desc + (uint64_t)((hl * (D * D * 2) + kk * 2048) >> 4), Cfg::IDESC_LIN,
                                       (hl > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit_warp(&bar[B_LIN_DONE + t]);
                    }
                }
                // drain: every MMA this thread issued has completed before the pair ends
                mma_commit_warp(&bar[B_DRAIN]);
                const uint32_t a = smem_u32(&bar[B_DRAIN]);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(a, 0)) {
                    if (globaltimer_ns() - t0 > p.wait_limit_ns) {
                        report_error(wc, HF_DEV_ERR_TIMEOUT, SITE_ATTN_DRAIN);
                        break;
                    }
                }
                if (!ok) *wc.abort_flag = 1;
            }
            __syncwarp();
            // ---- end of the pair ----
            tc_fence_before();
            const bool stop = bar_all_or(*wc.abort_flag != 0);
            tc_fence_after();
            if (stop) break;
            if (split) {
                P += R + kPartWeight;
                ++pair;
            } else {
                pair += gridDim.x;
            }
        }
    } else {
        // ======== warpgroups 1 and 2: softmax and epilogue of tile A / tile B ========
        reg_alloc<kRegsSoftmax>();
        const int t = (warp - 4) >> 2;
        int pair = pair_first;
        uint32_t P = pref_first;
        for (;;) {
            // this part of the pair (as in warpgroup 0, which finds its rounds)
            uint32_t R = 0;
            if (split) {
                if (pair >= p.total_pairs || P + kPartWeight >= e_c || s_c >= e_c) break;
                R = (uint32_t)p.pair_rounds[pair];
            } else if (pair >= p.total_pairs) {
                break;
            }
            int bh, qb0_[2], nblk_[2];
            pair_geometry(pair, bh, qb0_, nblk_);
            const int qb0 = t ? qb0_[1] : qb0_[0];     // this group's tile
            const int nblk = t ? nblk_[1] : nblk_[0];
            if (bar_all_or(*wc.abort_flag != 0)) break;   // list and barriers ready
            const int n_list = (int)misc[M_NLIST];
            const int n_rounds = (n_list + 1) / 2;
            // this part's rounds [ra, rb) of the pair's stream
            const int ra = (int)misc[M_RA];
            const int rb = min((int)misc[M_RB], n_rounds);
            const bool participated = (int)misc[M_LASTR + t] >= 0;   // in a round of this part
            if (nblk > 0) {
                const int quarter = warp & 3;            // TMEM lane quarter this warp may access
                const int r = quarter * 32 + lane;       // query row within the tile
                const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
                const uint32_t o_col = tmem + lane_addr + 256 * t;
                const uint32_t s_col = o_col + 128;
                const int gq = min(r / BETA, nblk - 1);   // the row's query block within the tile
                const float sl2 = g.scale_log2;
                float m_run = -INFINITY, m_use = -INFINITY;
                float lsum[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // partial row sums (independent chains)
                bool ok = true;
                int cnt = 0;
                // the next round this tile takes part in, and its list entries; looked
                // up right after P is handed over, while the next S is being computed
                uint32_t m_nx = 0, e_nx[2] = {0u, 0u};
                auto find_round = [&](int from) -> int {
                    int rr = from;
                    while (rr < rb && (m_nx = tile_bits(sCode[rr], t)) == 0u) ++rr;
                    if (rr < rb) {
                        e_nx[0] = sList[2 * rr + (m_nx == 2u ? 1 : 0)];
                        e_nx[1] = m_nx == 3u ? sList[2 * rr + 1] : 0u;
                    }
                    return rr;
                };
                for (int rd = find_round(ra); rd < rb; rd = find_round(rd + 1)) {
                    const int n = m_nx == 3u ? 2 : 1;
                    const uint32_t ent[2] = {e_nx[0], e_nx[1]};
                    // valid columns of this warp's rows in each slab: [0, lo) and [32, 32 + hi)
                    int lo[2] = {0, 0}, hi[2] = {0, 0};
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        if (i < n) {
                            const uint32_t e = ent[i];
                            const int slab = static_cast<int>(e & 0xFFFFu);
                            const int k = slab % p.spf;
                            const int nvs = min(64, g.nf - 64 * k);
                            const uint32_t mt = (e >> (16 + 8 * t)) & 0xFFu;
                            if (BETA >= 64) {
                                const int v = ((mt >> gq) & 1u) ? nvs : 0;
                                lo[i] = min(v, 32);
                                hi[i] = max(0, v - 32);
                            } else {
                                lo[i] = ((mt >> gq) & 1u) ? min(32, nvs) : 0;
                                hi[i] = ((mt >> (4 + gq)) & 1u) ? max(0, nvs - 32) : 0;
                            }
                        }
                    }
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[B_S_FULL + t], cnt & 1, wc, SITE_ATTN_S_FULL));
                    ++cnt;
                    if (!ok) break;
                    tc_fence_after();
                    const bool any = (lo[0] | hi[0] | lo[1] | hi[1]) != 0;
                    if (!any) {   // nothing of these slabs is selected for this warp's rows: P = 0
                        uint32_t zr[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c) zr[c] = 0u;
                        tmem_st16_nw(s_col, zr);
                        tmem_st16_nw(s_col + 16, zr);
                        if (n == 2) {
                            tmem_st16_nw(s_col + 32, zr);
                            tmem_st16_nw(s_col + 48, zr);
                        }
                        tmem_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar[B_P_FULL + t]);
                        continue;
                    }
                    uint32_t sr[4][32];
                    tmem_ld32_nw(s_col, sr[0]);
                    tmem_ld32_nw(s_col + 32, sr[1]);
                    if (n == 2) {
                        tmem_ld32_nw(s_col + 64, sr[2]);
                        tmem_ld32_nw(s_col + 96, sr[3]);
                    }
                    tmem_wait_ld();
                    reg_dep32(sr[0]);
                    reg_dep32(sr[1]);
                    if (n == 2) {
                        reg_dep32(sr[2]);
                        reg_dep32(sr[3]);
                    }
                    const bool full = lo[0] == 32 && hi[0] == 32 && (n == 1 || (lo[1] == 32 && hi[1] == 32));
                    if (!full) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            if (c >= lo[0]) sr[0][c] = 0xFF800000u;
                            if (c >= hi[0]) sr[1][c] = 0xFF800000u;
                            if (c >= lo[1]) sr[2][c] = 0xFF800000u;
                            if (c >= hi[1]) sr[3][c] = 0xFF800000u;
                        }
                    }
                    // row max over 8 independent chains
                    float mx[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) mx[q] = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        mx[(c >> 1) & 3] = fmax3(mx[(c >> 1) & 3], __uint_as_float(sr[0][c]), __uint_as_float(sr[0][c + 1]));
                        mx[4 + ((c >> 1) & 3)] =
                            fmax3(mx[4 + ((c >> 1) & 3)], __uint_as_float(sr[1][c]), __uint_as_float(sr[1][c + 1]));
                    }
                    if (n == 2) {
#pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            mx[(c >> 1) & 3] =
                                fmax3(mx[(c >> 1) & 3], __uint_as_float(sr[2][c]), __uint_as_float(sr[2][c + 1]));
                            mx[4 + ((c >> 1) & 3)] =
                                fmax3(mx[4 + ((c >> 1) & 3)], __uint_as_float(sr[3][c]), __uint_as_float(sr[3][c + 1]));
                        }
                    }
                    const float m_new =
                        fmax3(m_run, fmax3(mx[0], mx[1], fmax3(mx[2], mx[3], mx[4])), fmax3(mx[5], mx[6], mx[7]));
                    m_run = m_new;
                    // Lazy rescale: the exponent reference m_use only moves when the
                    // running max exceeds it by more than 8 (log2 units), so O and l
                    // stay consistent with m_use and p <= 2^8.  O_t is quiescent here:
                    // the commit that published S_t followed every earlier P V of the
                    // tile.  The TMEM access is warp-collective.
                    const bool move = m_use == -INFINITY || (m_new - m_use) * sl2 > 8.0f;
                    const bool scale_o = move && m_use != -INFINITY;
                    if (__any_sync(0xFFFFFFFFu, scale_o)) {
                        const float f = scale_o ? ex2_approx((m_use - m_new) * sl2) : 1.0f;
#pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t o[32];
                            tmem_ld32(o_col + c0, o);
#pragma unroll
                            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f);
                            tmem_st32(o_col + c0, o);
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q) lsum[q] *= f;
                    }
                    if (move) m_use = m_new;
                    const float neg = -m_use * sl2;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        if (h < 2 * n) {
                            uint32_t pk[16];
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                float a, b;
                                fma2(a, b, __uint_as_float(sr[h][2 * c]), __uint_as_float(sr[h][2 * c + 1]), sl2, sl2,
                                     neg, neg);
                                a = ex2_approx(a);
                                b = ex2_approx(b);
                                add2(lsum[(c & 1) * 2], lsum[(c & 1) * 2 + 1], lsum[(c & 1) * 2], lsum[(c & 1) * 2 + 1],
                                     a, b);
                                pk[c] = pack_bf16(a, b);
                            }
                            tmem_st16_nw(s_col + 16 * h, pk);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();   // the warp's P stores are complete: one arrival for the warp
                    if (lane == 0) mbar_arrive(&bar[B_P_FULL + t]);
                }
                if (ok && participated)
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[B_O_DONE + t], 0, wc, SITE_ATTN_PV_DONE));
                float l_tot = (lsum[0] + lsum[1]) + (lsum[2] + lsum[3]);
                // ---- a pair cut between CTAs: every part but the last to arrive leaves
                // (O, m, l) of each row in its slot; the part that arrives last merges all
                // parts in part order, its own from TMEM
                // (so the result does not depend on which part that is) and finishes
                // the pair ----
                bool do_out = true;
                // the same decision in all four warps: the protocol below has group barriers
                const bool gok = (FUSED && split) ? bar_group_and(2 + t, ok) : ok;
                if (FUSED && split && gok) {
                    const int G = gridDim.x;
                    // parts: the CTAs c0..c1 with a non-empty share (c0 and c1 own rounds,
                    // so their shares are never empty)
                    const uint32_t Pr = P + kPartWeight;   // unit of the pair's round 0
                    const int c0 = round_owner(Pr, T, G);
                    const int c1 = round_owner(Pr + R - 1, T, G);
                    int nparts = 0;
                    for (int c = c0; c <= c1; ++c) nparts += share_nonempty(c, T, G) ? 1 : 0;
                    if (nparts > 1) {
                        // CTA c's block, column-major (a warp's access to one column is one
                        // 128-byte line): c0 may also end an earlier pair, so it writes
                        // slot 1 when its share starts before this pair
                        auto part_col = [&](int c) -> float* {
                            const int slot = (c == c0 && share_start(c0, T, G) != Pr) ? 1 : 0;
                            return p.partial + (((size_t)c * 2 + slot) * 2 + t) * (size_t)((D + 4) * 128) + r;
                        };
                        const int me = (int)blockIdx.x;
                        float* mine = part_col(me);
                        const float m_own = participated ? m_use : -INFINITY;
                        const float l_own = participated ? l_tot : 0.0f;
                        if (participated) tc_fence_after();
                        // The head part of a pair (its round 0) ends its CTA's share, so it
                        // usually runs after the other parts, which start the following
                        // shares.  If they have all arrived, it is the last part: it merges
                        // without writing its own partial result.
                        bool all_in = false;
                        if (me == c0) {
                            if (r == 0) misc[M_OLD + t] = ld_acquire_gpu(p.counters + (size_t)pair * 2 + t);
                            asm volatile("bar.sync %0, 128;" ::"r"(2 + t) : "memory");
                            all_in = *reinterpret_cast<volatile uint32_t*>(&misc[M_OLD + t]) == (uint32_t)(nparts - 1);
                        }
                        if (!all_in) {
                            {   // the whole row at once: one TMEM round trip
                                uint32_t o[D / 32][32];
                                if (participated) {
#pragma unroll
                                    for (int cq = 0; cq < D / 32; ++cq) tmem_ld32_nw(o_col + 32 * cq, o[cq]);
                                    tmem_wait_ld();
#pragma unroll
                                    for (int cq = 0; cq < D / 32; ++cq) reg_dep32(o[cq]);
                                } else {
#pragma unroll
                                    for (int cq = 0; cq < D / 32; ++cq)
#pragma unroll
                                        for (int c = 0; c < 32; ++c) o[cq][c] = 0u;
                                }
#pragma unroll
                                for (int cq = 0; cq < D / 32; ++cq)
#pragma unroll
                                    for (int c = 0; c < 32; ++c)
                                        __stcg(mine + (32 * cq + c) * 128, __uint_as_float(o[cq][c]));
                            }
                            __stcg(mine + D * 128, m_own);
                            __stcg(mine + (D + 1) * 128, l_own);
                            asm volatile("bar.sync %0, 128;" ::"r"(2 + t) : "memory");
                            if (r == 0) {
                                __threadfence();
                                misc[M_OLD + t] = atomicAdd(p.counters + (size_t)pair * 2 + t, 1u);
                            }
                            asm volatile("bar.sync %0, 128;" ::"r"(2 + t) : "memory");
                        }
                        do_out = all_in ||
                                 *reinterpret_cast<volatile uint32_t*>(&misc[M_OLD + t]) == (uint32_t)(nparts - 1);
                        if (do_out && nparts == 2) {
                            // two parts (the usual cut): the other part's whole row is
                            // loaded at once (one memory round trip), then combined with
                            // this part's row from TMEM in part order (CTA order), with the
                            // same arithmetic as the general merge below
                            __threadfence();
                            const int oc = c0 == me ? c1 : c0;
                            const float* src = part_col(oc);
                            uint32_t vo[D / 32][32];
#pragma unroll
                            for (int cq = 0; cq < D / 32; ++cq)
#pragma unroll
                                for (int k = 0; k < 32; ++k) vo[cq][k] = __float_as_uint(__ldcg(src + (32 * cq + k) * 128));
                            const float mo = __ldcg(src + D * 128), lo = __ldcg(src + (D + 1) * 128);
                            const float m_all = fmaxf(m_own, mo);
                            auto scale_of = [&](float mk) { return mk == -INFINITY ? 0.0f : ex2_approx((mk - m_all) * sl2); };
                            const float sc_me = scale_of(m_own), sc_o = scale_of(mo);
                            const bool me_first = me < oc;
                            l_tot = me_first ? fmaf(sc_o, lo, fmaf(sc_me, l_own, 0.0f)) : fmaf(sc_me, l_own, fmaf(sc_o, lo, 0.0f));
#pragma unroll
                            for (int cq = 0; cq < D / 32; ++cq) {
                                uint32_t v[32];
                                if (participated) {
                                    tmem_ld32_nw(o_col + 32 * cq, v);
                                    tmem_wait_ld();
                                    reg_dep32(v);
                                } else {
#pragma unroll
                                    for (int k = 0; k < 32; ++k) v[k] = 0u;
                                }
#pragma unroll
                                for (int k = 0; k < 32; ++k) {
                                    const float own = __uint_as_float(v[k]), oth = __uint_as_float(vo[cq][k]);
                                    v[k] = __float_as_uint(me_first ? fmaf(sc_o, oth, fmaf(sc_me, own, 0.0f))
                                                                    : fmaf(sc_me, own, fmaf(sc_o, oth, 0.0f)));
                                }
                                tmem_st32(o_col + 32 * cq, v);
                            }
                            tc_fence_before();
                            if (r == 0) p.counters[(size_t)pair * 2 + t] = 0u;   // ready for the next launch
                        } else if (do_out) {
                            // merge in part order; this CTA's own part comes from TMEM
                            __threadfence();
                            float m_all = m_own;
                            for (int c = c0; c <= c1; ++c)
                                if (c != me && share_nonempty(c, T, G)) m_all = fmaxf(m_all, __ldcg(part_col(c) + D * 128));
                            auto scale_of = [&](float mk) { return mk == -INFINITY ? 0.0f : ex2_approx((mk - m_all) * sl2); };
                            const float sc_own = scale_of(m_own);
                            float lt = 0.0f;
#pragma unroll 1
                            for (int cb = 0; cb < D; cb += 32) {
                                float acc[32];
#pragma unroll
                                for (int c = 0; c < 32; ++c) acc[c] = 0.0f;
#pragma unroll 1
                                for (int c = c0; c <= c1; ++c) {
                                    if (!share_nonempty(c, T, G)) continue;
                                    float sc, lk;
                                    uint32_t v[32];
                                    if (c == me) {
                                        if (participated) {
                                            tmem_ld32_nw(o_col + cb, v);
                                            tmem_wait_ld();
                                            reg_dep32(v);
                                        } else {
#pragma unroll
                                            for (int k = 0; k < 32; ++k) v[k] = 0u;
                                        }
                                        sc = sc_own;
                                        lk = l_own;
                                    } else {
                                        const float* src = part_col(c);
#pragma unroll
                                        for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__ldcg(src + (cb + k) * 128));
                                        const float mk = __ldcg(src + D * 128);
                                        lk = __ldcg(src + (D + 1) * 128);
                                        sc = scale_of(mk);
                                    }
                                    if (cb == 0) lt = fmaf(sc, lk, lt);
#pragma unroll
                                    for (int k = 0; k < 32; ++k) acc[k] = fmaf(sc, __uint_as_float(v[k]), acc[k]);
                                }
                                uint32_t o[32];
#pragma unroll
                                for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(acc[k]);
                                tmem_st32(o_col + cb, o);
                            }
                            l_tot = lt;
                            tc_fence_before();
                            if (r == 0) p.counters[(size_t)pair * 2 + t] = 0u;   // ready for the next launch
                        }
                    }
                }
                const float inv_l = 1.0f / l_tot;
                if (FUSED) {
                    uint8_t* sQ = smem + Cfg::OFF_Q + t * Cfg::Q_BYTES;
                    if (ok && !do_out) {
                        // another part finishes this pair: the MMA thread skips its linear read
                        if (r == 0) misc[M_SKIPLIN + t] = 1u;
                        mbar_arrive(&bar[B_PHIQ + t]);
                    } else if (ok && (participated ||
                                      __all_sync(0xFFFFFFFFu, mbar_wait(&bar[B_Q], 0, wc, SITE_ATTN_Q)))) {
                        // (a tile that took part in no round of this part waits for its Q tile
                        // here; otherwise its S_FULL waits already covered the Q load)
                        tc_fence_after();
                        // phi(q) (bf16, in place over Q) and the linear-read denominator (z
                        // of the head from shared memory, four independent denominator
                        // chains), one 64-column chunk of the row per step.  Each step
                        // issues all its shared-memory loads (the row's eight 16-byte
                        // pieces and the chunk's 64 values of z) before using any: while
                        // the other tile's Q K^T keeps shared memory busy, every access
                        // waits long, and one round trip per chunk costs far less than one
                        // per piece.
                        const float4* zh = reinterpret_cast<const float4*>(smem + Cfg::OFF_Z);
                        float dn[4] = {g.eps, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
                        for (int h = 0; h < Cfg::DCH; ++h) {
                            uint8_t* rowp = sQ + h * (Cfg::TILE_M * 128) + r * 128;
                            uint4 qv[8];
                            float4 zv[16];
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                qv[j] = *reinterpret_cast<const uint4*>(rowp + (((j ^ (r & 7)) & 7) << 4));
#pragma unroll
                            for (int j = 0; j < 16; ++j) zv[j] = zh[16 * h + j];
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float zc[8] = {zv[2 * j].x,     zv[2 * j].y,     zv[2 * j].z,     zv[2 * j].w,
                                                     zv[2 * j + 1].x, zv[2 * j + 1].y, zv[2 * j + 1].z, zv[2 * j + 1].w};
                                uint32_t w4[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    float a = bf16_lo(w4[i]), bq = bf16_hi(w4[i]);
                                    a = phi_elu1(a);
                                    bq = phi_elu1(bq);
                                    w4[i] = pack_bf16(a, bq);
                                    dn[i] = fmaf(bf16_lo(w4[i]), zc[2 * i], dn[i]);
                                    dn[i] = fmaf(bf16_hi(w4[i]), zc[2 * i + 1], dn[i]);
                                }
                                *reinterpret_cast<uint4*>(rowp + (((j ^ (r & 7)) & 7) << 4)) =
                                    make_uint4(w4[0], w4[1], w4[2], w4[3]);
                            }
                        }
                        const float den = (dn[0] + dn[1]) + (dn[2] + dn[3]);
                        fence_proxy_async_smem();
                        tc_fence_before();
                        mbar_arrive(&bar[B_PHIQ + t]);
                        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[B_LIN_DONE + t], 0, wc, SITE_ATTN_LIN));
                        if (ok) {
                            tc_fence_after();
                            const float inv_den = 1.0f / den;
#pragma unroll 1
                            for (int cb = 0; cb < D; cb += 32) {
                                uint32_t o[32], li[32];
                                tmem_ld32_nw(o_col + cb, o);
                                tmem_ld32_nw(s_col + cb, li);
                                tmem_wait_ld();
                                reg_dep32(o);
                                reg_dep32(li);
                                uint8_t* rowp = sQ + (cb >> 6) * (Cfg::TILE_M * 128) + r * 128;
#pragma unroll
                                for (int cq = 0; cq < 4; ++cq) {   // 16-byte chunks of the row
                                    const int ch = ((cb >> 3) & 7) + cq;
                                    uint32_t w4[4];
#pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        const int c = cq * 8 + 2 * i;
                                        const float a =
                                            fmaf(__uint_as_float(o[c]), inv_l, __uint_as_float(li[c]) * inv_den);
                                        const float bq = fmaf(__uint_as_float(o[c + 1]), inv_l,
                                                              __uint_as_float(li[c + 1]) * inv_den);
                                        w4[i] = pack_bf16(a, bq);
                                    }
                                    *reinterpret_cast<uint4*>(rowp + (((ch ^ (r & 7)) & 7) << 4)) =
                                        make_uint4(w4[0], w4[1], w4[2], w4[3]);
                                }
                            }
                            fence_proxy_async_smem();
                        }
                    }
                    if (!ok) *wc.abort_flag = 1;
                    // every thread of this softmax group reaches this barrier exactly once
                    asm volatile("bar.sync %0, 128;" ::"r"(2 + t) : "memory");
                    if (r == 0 && *wc.abort_flag == 0 && do_out) {
                        for (int gb = 0; gb < nblk; ++gb) {
                            const int qbs = qb0 + gb;
                            const int cf = qbs / g.bpf;
                            const int js = qbs - cf * g.bpf;
                            for (int m = 0; m < Cfg::DCH; ++m)
                                tma_store_3d(&tmO, sQ + m * (Cfg::TILE_M * 128) + gb * BETA * 128, 64 * m, js * BETA,
                                             bh * g.C + cf);
                        }
                        bulk_commit();
                        bulk_wait_read_all();   // sQ is free again; the writes complete by the end
                    }
                } else if (ok) {
                    tc_fence_after();
                    const int qb = qb0 + gq;
                    const int c_frame = qb / g.bpf;
                    const int jq = qb - c_frame * g.bpf;
                    const int rin = r - gq * BETA;
                    const bool valid = (r / BETA) < nblk && rin < min(BETA, g.nf - jq * BETA);
                    float* dst =
                        p.o_swa + ((size_t)bh * g.C * g.nf + (size_t)c_frame * g.nf + (size_t)jq * BETA + rin) * D;
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(o_col + c0, o);
                        if (valid) {
#pragma unroll
                            for (int c = 0; c < 32; c += 4) {
                                float4 v4 = make_float4(
                                    __uint_as_float(o[c]) * inv_l, __uint_as_float(o[c + 1]) * inv_l,
                                    __uint_as_float(o[c + 2]) * inv_l, __uint_as_float(o[c + 3]) * inv_l);
                                *reinterpret_cast<float4*>(dst + c0 + c) = v4;
                            }
                        }
                    }
                }
                // keep the MMA thread from waiting on arrivals that will not come
                if (!ok) *wc.abort_flag = 1;
            }
            // ---- end of the pair ----
            tc_fence_before();
            const bool stop = bar_all_or(*wc.abort_flag != 0);
            tc_fence_after();
            if (stop) break;
            if (split) {
                P += R + kPartWeight;
                ++pair;
            } else {
                pair += gridDim.x;
            }
        }
    }
    if (warp >= 4 && (warp & 3) == 0 && lane == 0) bulk_wait_all();   // the output stores of this CTA
    tc_fence_before();
    bar_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

template <int D, int BETA, bool FUSED>
int launch_attn_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                  const AttnParams& p, int grid, cudaStream_t st)
{
    using Cfg = AttnCfg<D, BETA>;
    auto kern = attn_kernel<D, BETA, FUSED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC);
    if (e != cudaSuccess) return (int)e;
    kern<<<grid, kThreads, Cfg::SMEM_ALLOC, st>>>(tq, tk, tv, to, p);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_attn(const uint16_t* Q, const uint16_t* Kc, const uint16_t* Vc, const Geom& g, const SlotMap& sm,
                const int32_t* idx, const uint16_t* smma, const float* z, float* o_swa, uint16_t* o_bf16,
                const int32_t* pair_rounds, float* partial, uint32_t* counters, uint32_t* status,
                uint64_t wait_limit_ns, void* stream)
{
    const bool fused = o_bf16 != nullptr;
    const int qrows = g.beta;   // Q / O box rows = one query block
    alignas(64) CUtensorMap tq, tk, tv, to;
    int e;
    // Q and O: [BH*C planes][nf rows][d]; K, V: [BH*W slots][nf valid rows][d], slot pitch slot_stride rows
    e = make_tmap_bf16_3d(&tq, Q, g.d, g.nf, (uint64_t)g.BH * g.C, (uint64_t)g.d * 2, (uint64_t)g.nf * g.d * 2, 64,
                          qrows);
    if (e) return e;
    e = make_tmap_bf16_3d(&tk, Kc, g.d, g.nf, (uint64_t)g.BH * g.W, (uint64_t)g.d * 2,
                          (uint64_t)g.slot_stride * g.d * 2, 64, 64);
    if (e) return e;
    e = make_tmap_bf16_3d(&tv, Vc, g.d, g.nf, (uint64_t)g.BH * g.W, (uint64_t)g.d * 2,
                          (uint64_t)g.slot_stride * g.d * 2, 64, 64);
    if (e) return e;
    if (fused) {
        e = make_tmap_bf16_3d(&to, o_bf16, g.d, g.nf, (uint64_t)g.BH * g.C, (uint64_t)g.d * 2,
                              (uint64_t)g.nf * g.d * 2, 64, qrows);
        if (e) return e;
    } else {
        to = tq;
    }
    AttnParams p;
    p.g = g;
    p.sm = sm;
    p.idx = idx;
    p.smma = smma;
    p.z = z;
    p.o_swa = o_swa;
    p.status = status;
    p.wait_limit_ns = wait_limit_ns;
    const int G = 128 / g.beta;
    p.tiles_per_head = (g.nqb + G - 1) / G;
    p.pairs_per_head = (p.tiles_per_head + 1) / 2;
    p.total_pairs = g.BH * p.pairs_per_head;
    p.spf = (g.nf + 63) / 64;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // split mode (fused forward with the prologue's pair weights): one CTA per
    // SM, each an equal share of all pairs' weighted rounds; otherwise whole pairs
    // in turn
    const bool split = fused && pair_rounds && partial && counters;
    p.pair_rounds = split ? pair_rounds : nullptr;
    p.partial = split ? partial : nullptr;
    p.counters = split ? counters : nullptr;
    const int grid = split ? (sms < kAttnMaxGrid ? sms : kAttnMaxGrid) : (p.total_pairs < sms ? p.total_pairs : sms);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
#define HF_ATTN_CASE(DD, BB)                                                                       \
    if (g.d == DD && g.beta == BB)                                                                 \
        return fused ? launch_attn_t<DD, BB, true>(tq, tk, tv, to, p, grid, st)                    \
                     : launch_attn_t<DD, BB, false>(tq, tk, tv, to, p, grid, st);
    HF_ATTN_CASE(128, 64)
    HF_ATTN_CASE(128, 128)
    HF_ATTN_CASE(128, 32)
    HF_ATTN_CASE(64, 32)
    HF_ATTN_CASE(64, 64)
    HF_ATTN_CASE(64, 128)
#undef HF_ATTN_CASE
    return (int)cudaErrorInvalidValue;
}

}  // namespace hf
