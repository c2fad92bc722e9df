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
// tiles of one head (A and B) in turn.  The two tiles share one stream of
// slabs -- the union of both tiles' slabs in window order -- so a slab that
// both need is loaded once.  The stream is cut into rounds of two slabs; a
// tile takes part in a round when it needs one or both of its slabs.  The
// two slabs of a round sit one above the other in shared memory, so when a
// tile needs both, Q K^T is one N = 128 MMA per K step (an N = 64 MMA reads
// as many operand bytes from shared memory per FLOP as it computes, and runs
// at about half the tensor core's rate).
//
// Warp roles (384 threads = 3 warpgroups, 1 CTA per SM):
//   warps 0-3  build the pair's slab stream; then
//   warp 0     TMA producer of the Q tiles, of the keys (a ring of NR round
//              stages) and, at the end, of the bf16 hi/lo state S for the
//              fused linear read (into the key ring);
//   warp 2     TMA producer of the values (a second ring of NR round stages).
//              Keys are released as soon as Q K^T has read them, values
//              after P V: each ring runs about NR rounds ahead.
//   warp 1     TMEM owner + single-thread MMA issuer, in the order
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
    static constexpr int SMEM = OFF_MISC + 128;
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
    B_K_FULL = 1,      // 4 (NR)
    B_K_EMPTY = 5,     // 4
    B_V_FULL = 9,      // 4
    B_V_EMPTY = 13,    // 4
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
enum { M_TMEM = 0, M_ABORT = 1, M_NLIST = 2, M_LAST = 3 /* 2 */, M_WCOUNT = 8 /* 4 */ };

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
};

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
// of the stream, in order, each into the stage of its round.  Returns the
// number of rounds issued; *ok = false if a wait gave up.
template <int D, int BETA>
__device__ __forceinline__ int produce_ring(const CUtensorMap* tm, uint8_t* ring, uint64_t* full, uint64_t* empty,
                                            const uint32_t* list, int n_list, int n_rounds, int bh,
                                            const AttnParams& p, const WaitCtl& wc, uint32_t site, bool& ok)
{
    using Cfg = AttnCfg<D, BETA>;
    int r = 0;
    for (; r < n_rounds; ++r) {
        const int s = r % Cfg::NR;
        if (r >= Cfg::NR && !mbar_wait(&empty[s], ((r / Cfg::NR) - 1) & 1, wc, site)) {
            ok = false;
            break;
        }
        const int nq = min(2, n_list - 2 * r);
        uint8_t* st = ring + s * Cfg::RS_BYTES;
        mbar_arrive_expect_tx(&full[s], nq * Cfg::SLAB_BYTES);
        for (int i = 0; i < nq; ++i) {
            const int slab = static_cast<int>(list[2 * r + i] & 0xFFFFu);
            const int w = slab / p.spf;
            const int k = slab - w * p.spf;
            const int plane = bh * p.g.W + p.sm.s[w];
            for (int m = 0; m < Cfg::DCH; ++m)
                tma_load_3d(st + m * Cfg::CHUNK + i * (Cfg::SLAB * 128), tm, &full[s], 64 * m, 64 * k, plane);
        }
    }
    return r;
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
        for (int pair = blockIdx.x; pair < p.total_pairs; pair += gridDim.x) {
            int bh, qb0[2], nblk[2];
            pair_geometry(pair, bh, qb0, nblk);
            // ---- barriers (no asynchronous operation is pending here) ----
            if (tid == 0) {
                mbar_init(&bar[B_Q], 1);
                for (int s = 0; s < Cfg::NR; ++s) {
                    mbar_init(&bar[B_K_FULL + s], 1);
                    mbar_init(&bar[B_K_EMPTY + s], 1);
                    mbar_init(&bar[B_V_FULL + s], 1);
                    mbar_init(&bar[B_V_EMPTY + s], 1);
                }
                for (int t = 0; t < 2; ++t) {
                    mbar_init(&bar[B_S_FULL + t], 1);
                    mbar_init(&bar[B_P_FULL + t], 128);
                    mbar_init(&bar[B_O_DONE + t], 1);
                    mbar_init(&bar[B_PHIQ + t], 128);
                    mbar_init(&bar[B_LIN_DONE + t], 1);
                }
                mbar_init(&bar[B_LIN_FULL], 1);
                mbar_init(&bar[B_DRAIN], 1);
                misc[M_LAST] = 0;
                misc[M_LAST + 1] = 0;
                fence_mbar_init();
            }
            // ---- the pair's slab stream ----
            // mask bits of slab s: tile t, sub-block h (beta = 32 only), query
            // block gq of the tile -> bit 8t + 4h + gq.
            const int nsl = g.n_win * p.spf;
            for (int i = tid; i < (nsl + 1) / 2; i += 128) sMask[i] = 0;
            bar_ctl();
            for (int t = 0; t < 2; ++t) {
                const int total = nblk[t] * g.k_eff;
                const int32_t* ip = p.idx + ((size_t)bh * g.nqb + qb0[t]) * g.k_eff;
                for (int i = tid; i < total; i += 128) {
                    const int gq = i / g.k_eff;
                    const int kb = ip[i];
                    if (kb < 0 || kb >= g.nkb) {
                        report_error(wc, HF_DEV_ERR_CHECK, SITE_ATTN_BAD_INDEX);
                        continue;
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
                }
            }
            bar_ctl();
            {   // ordered compaction of the slabs that either tile needs
                int base_out = 0;
                for (int base = 0; base < nsl; base += 128) {
                    const int s = base + tid;
                    const uint32_t m = s < nsl ? (sMask[s >> 1] >> ((s & 1) * 16)) & 0xFFFFu : 0u;
                    const uint32_t ball = __ballot_sync(0xFFFFFFFFu, m != 0);
                    if (lane == 0) misc[M_WCOUNT + warp] = __popc(ball);
                    bar_ctl();
                    int before = base_out, tot = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int c = (int)misc[M_WCOUNT + q];
                        if (q < warp) before += c;
                        tot += c;
                    }
                    if (m != 0) {
                        const int pos = before + __popc(ball & ((1u << lane) - 1u));
                        sList[pos] = static_cast<uint32_t>(s) | (m << 16);
                        if (m & 0x00FFu) atomicMax(&misc[M_LAST + 0], (uint32_t)pos + 1u);
                        if (m & 0xFF00u) atomicMax(&misc[M_LAST + 1], (uint32_t)pos + 1u);
                    }
                    base_out += tot;
                    bar_ctl();
                }
                if (tid == 0) misc[M_NLIST] = base_out;
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
            }
            // list and barriers ready; a bad index: nothing of this pair is issued
            if (bar_all_or(*wc.abort_flag != 0)) break;
            const int n_list = (int)misc[M_NLIST];
            const int n_rounds = (n_list + 1) / 2;

            if (warp == 0 && lane == 0) {
                // ---------- Q tiles, key ring, state operand ----------
                bool ok = true;
                const int ntiles = (nblk[0] > 0) + (nblk[1] > 0);
                mbar_arrive_expect_tx(&bar[B_Q], ntiles * Cfg::G * Cfg::DCH * BETA * 128);
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
                const int issued = produce_ring<D, BETA>(&tmK, sK, &bar[B_K_FULL], &bar[B_K_EMPTY], sList, n_list,
                                                         n_rounds, bh, p, wc, SITE_ATTN_KV_EMPTY, ok);
                bool lin_issued = false;
                if (FUSED && ok) {
                    // the state operands go into the key ring once every key stage is free
                    for (int r = max(0, n_rounds - Cfg::NR); r < n_rounds && ok; ++r)
                        ok = mbar_wait(&bar[B_K_EMPTY + r % Cfg::NR], (r / Cfg::NR) & 1, wc, SITE_ATTN_KV_EMPTY);
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
                for (int r = max(0, issued - Cfg::NR); r < issued; ++r)
                    drain_wait(&bar[B_K_FULL + r % Cfg::NR], (r / Cfg::NR) & 1, p.wait_limit_ns);
                drain_wait(&bar[B_Q], 0, p.wait_limit_ns);
                if (lin_issued) drain_wait(&bar[B_LIN_FULL], 0, p.wait_limit_ns);
                if (!ok) *wc.abort_flag = 1;
            } else if (warp == 2 && lane == 0) {
                // ---------- value ring ----------
                bool ok = true;
                const int issued = produce_ring<D, BETA>(&tmV, sV, &bar[B_V_FULL], &bar[B_V_EMPTY], sList, n_list,
                                                         n_rounds, bh, p, wc, SITE_ATTN_KV_EMPTY, ok);
                for (int r = max(0, issued - Cfg::NR); r < issued; ++r)
                    drain_wait(&bar[B_V_FULL + r % Cfg::NR], (r / Cfg::NR) & 1, p.wait_limit_ns);
                if (!ok) *wc.abort_flag = 1;
            } else if (warp == 1 && lane == 0) {
                // ---------- MMA issuer ----------
                // Batches in the order A(-1) B(-1) A(0) B(0) A(1) ..., batch t(r) =
                // P V_t(r) followed by Q K^T_t(r+1) (S_t is free again once P V_t(r) has
                // been issued: the tensor core executes in issue order).  Each tile's
                // softmax then runs while the tensor core works on the other tile's
                // batch.  The MMA queue holds only a few MMAs, so the thread keeps the
                // work between batches short: round codes are read ahead, and each
                // round's key and value stages are waited for once.
                bool ok = mbar_wait(&bar[B_Q], 0, wc, SITE_ATTN_Q);
                tc_fence_after();
                // base descriptors (start addresses advance in 16-byte units): Q tiles and
                // the key ring K-major, the value ring MN-major (64-column chunks CHUNK apart)
                const uint64_t q_desc0 = smem_desc(smem_u32(smem + Cfg::OFF_Q), 16, 1024);
                const uint64_t q_desc1 = smem_desc(smem_u32(smem + Cfg::OFF_Q + Cfg::Q_BYTES), 16, 1024);
                const uint64_t k_desc = smem_desc(smem_u32(sK), 16, 1024);
                const uint64_t v_desc = smem_desc(smem_u32(sV), Cfg::CHUNK, 1024);
                const int last_round0 = ((int)misc[M_LAST + 0] - 1) >> 1;
                const int last_round1 = ((int)misc[M_LAST + 1] - 1) >> 1;
                int cnt0 = 0, cnt1 = 0;
                bool first0 = true, first1 = true;
                int k_round = -1, v_round = -1;   // last round whose key / value stage was waited for
                // m: the tile's slabs of round r (bit i = slab i), from the round code
                auto issue_qk = [&](int r, int t, uint32_t m) -> bool {
                    if (m == 0) return true;
                    const int s = r % Cfg::NR;
                    if (r > k_round) {
                        if (!mbar_wait(&bar[B_K_FULL + s], (r / Cfg::NR) & 1, wc, SITE_ATTN_KV_FULL)) return false;
                        k_round = r;
                    }
                    tc_fence_after();
                    const uint64_t qd = t ? q_desc1 : q_desc0;
                    // both slabs: one N = 128 operand; one slab: its 64 rows
                    const uint64_t kd =
                        k_desc + (uint64_t)((s * Cfg::RS_BYTES + (m == 2u ? Cfg::SLAB * 128 : 0)) >> 4);
                    const uint32_t idesc = m == 3u ? Cfg::IDESC_QK128 : Cfg::IDESC_QK64;
                    const uint32_t dt = tmem + 256 * t + 128;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(dt, qd + (uint64_t)(((kk >> 2) * (Cfg::TILE_M * 128) + (kk & 3) * 32) >> 4),
                               kd + (uint64_t)(((kk >> 2) * Cfg::CHUNK + (kk & 3) * 32) >> 4), idesc, kk > 0 ? 1u : 0u);
                    mma_commit(&bar[B_S_FULL + t]);
                    return true;
                };
                auto issue_pv = [&](int r, int t, uint32_t m) -> bool {
                    if (m == 0) return true;
                    int& cnt = t ? cnt1 : cnt0;
                    bool& first = t ? first1 : first0;
                    if (!mbar_wait(&bar[B_P_FULL + t], cnt & 1, wc, SITE_ATTN_P_FULL)) return false;
                    ++cnt;
                    const int s = r % Cfg::NR;
                    if (r > v_round) {
                        if (!mbar_wait(&bar[B_V_FULL + s], (r / Cfg::NR) & 1, wc, SITE_ATTN_KV_FULL)) return false;
                        v_round = r;
                    }
                    tc_fence_after();
                    const int n = m == 3u ? 2 : 1;
                    const uint32_t o_tm = tmem + 256 * t;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        if (j >= n) break;
                        const int i = (m == 2u) ? 1 : j;   // slab of the round; P columns [32j, 32j + 32)
                        const uint64_t vd = v_desc + (uint64_t)((s * Cfg::RS_BYTES + i * Cfg::SLAB * 128) >> 4);
                        const uint32_t at = o_tm + 128 + 32 * j;
#pragma unroll
                        for (int kk = 0; kk < Cfg::SLAB / 16; ++kk)
                            mma_ts(o_tm, at + kk * 8, vd + (uint64_t)(kk * (2048 >> 4)), Cfg::IDESC_PV,
                                   (first && j == 0 && kk == 0) ? 0u : 1u);
                    }
                    first = false;
                    if (r == (t ? last_round1 : last_round0)) mma_commit(&bar[B_O_DONE + t]);
                    return true;
                };
                // round codes are read one round ahead of their use
                uint32_t c_cur = sCode[0];
                uint32_t c_nxt = n_rounds > 1 ? sCode[1] : 0u;
                if (ok) ok = issue_qk(0, 0, tile_bits(c_cur, 0)) && issue_qk(0, 1, tile_bits(c_cur, 1));
                if (ok) mma_commit(&bar[B_K_EMPTY + 0]);
                for (int r = 0; ok && r < n_rounds; ++r) {
                    const uint32_t c_nn = r + 2 < n_rounds ? sCode[r + 2] : 0u;
                    const bool more = r + 1 < n_rounds;
                    ok = issue_pv(r, 0, tile_bits(c_cur, 0));
                    if (ok && more) ok = issue_qk(r + 1, 0, tile_bits(c_nxt, 0));
                    if (ok) ok = issue_pv(r, 1, tile_bits(c_cur, 1));
                    if (!ok) break;
                    mma_commit(&bar[B_V_EMPTY + r % Cfg::NR]);
                    if (more) {
                        ok = issue_qk(r + 1, 1, tile_bits(c_nxt, 1));
                        if (ok) mma_commit(&bar[B_K_EMPTY + (r + 1) % Cfg::NR]);
                    }
                    c_cur = c_nxt;
                    c_nxt = c_nn;
                }
                if (FUSED && ok) {
                    ok = mbar_wait(&bar[B_LIN_FULL], 0, wc, SITE_ATTN_LIN);
                    const uint64_t l_desc = smem_desc(smem_u32(sK), D * 128, 1024);
                    for (int t = 0; ok && t < 2; ++t) {
                        if (nblk[t] == 0) continue;
                        ok = mbar_wait(&bar[B_PHIQ + t], 0, wc, SITE_ATTN_PHIQ);
                        if (!ok) break;
                        tc_fence_after();
                        const uint64_t qd = t ? q_desc1 : q_desc0;
#pragma unroll
                        for (int hl = 0; hl < 2; ++hl) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_ss(tmem + 256 * t + 128,
                                       qd + (uint64_t)(((kk >> 2) * (Cfg::TILE_M * 128) + (kk & 3) * 32) >> 4),
                                       l_desc + (uint64_t)((hl * (D * D * 2) + kk * 2048) >> 4), Cfg::IDESC_LIN,
                                       (hl > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&bar[B_LIN_DONE + t]);
                    }
                }
                // drain: every MMA this thread issued has completed before the pair ends
                mma_commit(&bar[B_DRAIN]);
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
        }
    } else {
        // ======== warpgroups 1 and 2: softmax and epilogue of tile A / tile B ========
        reg_alloc<kRegsSoftmax>();
        const int t = (warp - 4) >> 2;
        for (int pair = blockIdx.x; pair < p.total_pairs; pair += gridDim.x) {
            int bh, qb0_[2], nblk_[2];
            pair_geometry(pair, bh, qb0_, nblk_);
            const int qb0 = t ? qb0_[1] : qb0_[0];     // this group's tile
            const int nblk = t ? nblk_[1] : nblk_[0];
            if (bar_all_or(*wc.abort_flag != 0)) break;   // list and barriers ready
            const int n_list = (int)misc[M_NLIST];
            const int n_rounds = (n_list + 1) / 2;
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
                    while (rr < n_rounds && (m_nx = tile_bits(sCode[rr], t)) == 0u) ++rr;
                    if (rr < n_rounds) {
                        e_nx[0] = sList[2 * rr + (m_nx == 2u ? 1 : 0)];
                        e_nx[1] = m_nx == 3u ? sList[2 * rr + 1] : 0u;
                    }
                    return rr;
                };
                for (int rd = find_round(0); rd < n_rounds; rd = find_round(rd + 1)) {
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
                        mbar_arrive(&bar[B_P_FULL + t]);
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
                    mbar_arrive(&bar[B_P_FULL + t]);
                }
                if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[B_O_DONE + t], 0, wc, SITE_ATTN_PV_DONE));
                const float inv_l = 1.0f / ((lsum[0] + lsum[1]) + (lsum[2] + lsum[3]));
                if (FUSED) {
                    uint8_t* sQ = smem + Cfg::OFF_Q + t * Cfg::Q_BYTES;
                    if (ok) {
                        tc_fence_after();
                        // phi(q) (bf16, in place over Q) and the linear-read denominator
                        const float* zh = p.z + (size_t)bh * D;
                        float den = g.eps;
#pragma unroll
                        for (int m = 0; m < Cfg::DCH; ++m) {
                            uint8_t* rowp = sQ + m * (Cfg::TILE_M * 128) + r * 128;
#pragma unroll
                            for (int ch = 0; ch < 8; ++ch) {
                                uint4* ptr = reinterpret_cast<uint4*>(rowp + (((ch ^ (r & 7)) & 7) << 4));
                                uint4 v = *ptr;
                                uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int c = m * 64 + ch * 8 + 2 * i;
                                    float a = bf16_lo(w4[i]), bq = bf16_hi(w4[i]);
                                    a = a > 0.0f ? a + 1.0f : __expf(a);
                                    bq = bq > 0.0f ? bq + 1.0f : __expf(bq);
                                    w4[i] = pack_bf16(a, bq);
                                    den = fmaf(bf16_lo(w4[i]), __ldg(zh + c), den);
                                    den = fmaf(bf16_hi(w4[i]), __ldg(zh + c + 1), den);
                                }
                                *ptr = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                            }
                        }
                        fence_proxy_async_smem();
                        tc_fence_before();
                        mbar_arrive(&bar[B_PHIQ + t]);
                        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[B_LIN_DONE + t], 0, wc, SITE_ATTN_LIN));
                        if (ok) {
                            tc_fence_after();
                            const float inv_den = 1.0f / den;
#pragma unroll
                            for (int c0 = 0; c0 < D; c0 += 32) {
                                uint32_t o[32], li[32];
                                tmem_ld32_nw(o_col + c0, o);
                                tmem_ld32_nw(s_col + c0, li);
                                tmem_wait_ld();
                                reg_dep32(o);
                                reg_dep32(li);
                                uint8_t* rowp = sQ + (c0 >> 6) * (Cfg::TILE_M * 128) + r * 128;
#pragma unroll
                                for (int ch = 0; ch < 4; ++ch) {
                                    uint32_t w4[4];
#pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        const int c = ch * 8 + 2 * i;
                                        const float a =
                                            fmaf(__uint_as_float(o[c]), inv_l, __uint_as_float(li[c]) * inv_den);
                                        const float bq = fmaf(__uint_as_float(o[c + 1]), inv_l,
                                                              __uint_as_float(li[c + 1]) * inv_den);
                                        w4[i] = pack_bf16(a, bq);
                                    }
                                    const int lch = ((c0 & 63) >> 3) + ch;   // logical 16-byte chunk of the row
                                    *reinterpret_cast<uint4*>(rowp + (((lch ^ (r & 7)) & 7) << 4)) =
                                        make_uint4(w4[0], w4[1], w4[2], w4[3]);
                                }
                            }
                            fence_proxy_async_smem();
                        }
                    }
                    if (!ok) *wc.abort_flag = 1;
                    // every thread of this softmax group reaches this barrier exactly once
                    asm volatile("bar.sync %0, 128;" ::"r"(2 + t) : "memory");
                    if (r == 0 && *wc.abort_flag == 0) {
                        for (int gb = 0; gb < nblk; ++gb) {
                            const int qbs = qb0 + gb;
                            const int cf = qbs / g.bpf;
                            const int js = qbs - cf * g.bpf;
                            for (int m = 0; m < Cfg::DCH; ++m)
                                tma_store_3d(&tmO, sQ + m * (Cfg::TILE_M * 128) + gb * BETA * 128, 64 * m, js * BETA,
                                             bh * g.C + cf);
                        }
                        bulk_commit();
                        bulk_wait_all();
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
        }
    }
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
                uint32_t* status, uint64_t wait_limit_ns, void* stream)
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
    const int grid = p.total_pairs < sms ? p.total_pairs : sms;
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
