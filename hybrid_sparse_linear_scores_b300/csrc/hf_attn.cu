// hf_attn.cu -- block-sparse sliding-window softmax attention on tcgen05,
// with the linear-read + sum epilogue fused in (Hybrid Forcing, English
// technical summary, section 2.A.2 "Block-Sparse Sliding Window Attention"
// and section 2.A.1 "Linear Temporal Attention"; the output is the sum of
// both paths, Spanish technical summary, section 2.A).
//
// One CTA owns a tile of 128 query rows = G = 128/beta consecutive query
// blocks of one head.  It attends to the UNION of their selected key blocks;
// for a row whose own block did not select a key block, that block's logits
// are masked to -inf, so every row sees exactly its own selection.
//
// Warp roles (192 threads, 2 CTAs per SM):
//   warp 0     TMA producer: Q tile once, then per 64-key unit the K and V
//              rows of the selected blocks, gathered from the frame ring
//              (2 stages); finally the bf16 hi/lo state S for the linear read.
//   warp 1     TMEM owner + single-thread MMA issuer:
//                S_u  = Q K_u^T      (SS MMA, M=128 N=64, K = d)
//                O   += P_u V_u      (TS MMA, P read from TMEM, N = d)
//                LIN  = phi(Q) S_hi + phi(Q) S_lo   (fused epilogue)
//   warps 2-5  softmax: one TMEM lane (= query row) per thread; online
//              softmax in fp32 with exp2, lazy rescale of O (only when the
//              running max grows by more than 2^8), P written back to TMEM
//              as bf16; epilogue O/l + LIN/(phi(q).z + eps) -> bf16 -> TMA store.
// TMEM columns: O [0, d), S/P buffers [d, d+64) and [d+64, d+128); LIN
// reuses the S/P columns after the last unit.
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

template <int D, int BETA>
struct AttnCfg {
    static constexpr int TILE_M = 128;
    static constexpr int G = 128 / BETA;               // query blocks per tile
    static constexpr int UNIT = 64;                    // keys per pipeline unit
    static constexpr int SUB = BETA < 64 ? BETA : 64;  // rows per K/V TMA box
    static constexpr int SEGS = UNIT / SUB;            // boxes per unit (2 for beta 32)
    static constexpr int DCH = D / 64;                 // 64-column chunks
    static constexpr int NS = 2;                       // K/V stages
    static constexpr int Q_BYTES = TILE_M * D * 2;
    static constexpr int KV_BYTES = UNIT * D * 2;
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    static constexpr int LIN_BYTES = 2 * D * D * 2;    // S hi + lo (bf16)
    static_assert(LIN_BYTES <= NS * STAGE_BYTES, "state operands must fit in the stage buffers");
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_STAGE = Q_BYTES;
    static constexpr int OFF_UNION = OFF_STAGE + NS * STAGE_BYTES;       // uint32[HF_MAX_KEY_BLOCKS]
    static constexpr int OFF_SEL = OFF_UNION + 4 * HF_MAX_KEY_BLOCKS;    // uint32[HF_MAX_KEY_BLOCKS/4]
    static constexpr int OFF_BAR = OFF_SEL + HF_MAX_KEY_BLOCKS;          // mbarriers
    static constexpr int NBAR = 16;
    static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;                  // tmem base, abort, counts
    static constexpr int SMEM = OFF_MISC + 64;
    static constexpr int SMEM_ALLOC = SMEM + 1024;                       // slack for 1 KB alignment
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr uint32_t O_COL = 0;
    static constexpr uint32_t S_COL = D;
    static constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, UNIT, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, false, true);
    static constexpr uint32_t IDESC_LIN = idesc_bf16_f32(128, D, false, true);
};

// barrier slots
enum { B_Q = 0, B_KV_FULL = 1, B_KV_EMPTY = 3, B_S_FULL = 5, B_P_FULL = 7, B_PV_DONE = 9, B_LIN_FULL = 11,
       B_PHIQ = 12, B_LIN_DONE = 13, B_DRAIN = 14 };

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
};

// One pipeline unit = 64 key rows from one (beta >= 64) or two (beta = 32)
// key blocks.  Every role walks the same unit sequence.
struct Seg {
    int kb;          // key block index (logical window order)
    uint32_t sel;    // bit g set: query block g of the tile selected kb
    int y;           // first row of the box inside the frame
    int nv;          // valid rows in the box (0..SUB)
};

template <int D, int BETA>
struct UnitWalk {
    using Cfg = AttnCfg<D, BETA>;
    const uint32_t* U;
    int nU, bpf, nf;
    int e = 0, half = 0;

    __device__ __forceinline__ UnitWalk(const uint32_t* u, int n, int b, int f) : U(u), nU(n), bpf(b), nf(f) {}

    __device__ __forceinline__ bool done() const { return e >= nU; }

    __device__ __forceinline__ Seg seg_of(int entry, int h) const
    {
        const uint32_t w = U[entry];
        Seg s;
        s.kb = static_cast<int>(w & 0xFFFFu);
        s.sel = w >> 16;
        const int j = s.kb % bpf;
        s.y = j * BETA + h * 64;
        const int rows = min(BETA, nf - j * BETA) - h * 64;
        s.nv = max(0, min(Cfg::SUB, rows));
        return s;
    }

    // Fills seg[0..SEGS) for the current unit and advances.
    __device__ __forceinline__ void next(Seg (&seg)[2])
    {
        if (BETA == 32) {
            seg[0] = seg_of(e, 0);
            if (e + 1 < nU) {
                seg[1] = seg_of(e + 1, 0);
            } else {   // odd count: load the first block again, mask it out
                seg[1] = seg[0];
                seg[1].sel = 0;
            }
            e += 2;
        } else if (BETA == 64) {
            seg[0] = seg_of(e, 0);
            seg[1] = seg[0];
            e += 1;
        } else {   // BETA == 128: two halves, skip an empty second half
            seg[0] = seg_of(e, half);
            seg[1] = seg[0];
            const int j = seg[0].kb % bpf;
            const bool has_second = (nf - j * BETA) > 64;
            if (half == 0 && has_second) {
                half = 1;
            } else {
                half = 0;
                e += 1;
            }
        }
    }
};

template <int D, int BETA>
__device__ __forceinline__ int count_units(const uint32_t* U, int nU, int bpf, int nf)
{
    if (BETA == 32) return (nU + 1) / 2;
    if (BETA == 64) return nU;
    int n = 0;
    for (int e = 0; e < nU; ++e) {
        const int j = static_cast<int>(U[e] & 0xFFFFu) % bpf;
        n += (nf - j * BETA) > 64 ? 2 : 1;
    }
    return n;
}

template <int D, int BETA, bool FUSED>
__global__ void __launch_bounds__(192, 2)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                const AttnParams p)
{
    using Cfg = AttnCfg<D, BETA>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + Cfg::OFF_Q;
    uint8_t* sStage = smem + Cfg::OFF_STAGE;
    uint32_t* sUnion = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_UNION);
    uint32_t* sSel = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_SEL);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
    // misc[0] tmem base, misc[1] abort flag, misc[2] union count, misc[3..6] warp partial counts

    const Geom& g = p.g;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int bh = blockIdx.x / p.tiles_per_head;
    const int tile = blockIdx.x - bh * p.tiles_per_head;
    const int qb0 = tile * Cfg::G;
    const int nblk = min(Cfg::G, g.nqb - qb0);

    WaitCtl wc{reinterpret_cast<volatile uint32_t*>(misc + 1), p.status, p.wait_limit_ns};

    if (tid == 0) {
        mbar_init(&bar[B_Q], 1);
        for (int s = 0; s < Cfg::NS; ++s) {
            mbar_init(&bar[B_KV_FULL + s], 1);
            mbar_init(&bar[B_KV_EMPTY + s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bar[B_S_FULL + b], 1);
            mbar_init(&bar[B_P_FULL + b], 128);
            mbar_init(&bar[B_PV_DONE + b], 1);
        }
        mbar_init(&bar[B_LIN_FULL], 1);
        mbar_init(&bar[B_PHIQ], 128);
        mbar_init(&bar[B_LIN_DONE], 1);
        mbar_init(&bar[B_DRAIN], 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        if (FUSED) prefetch_tmap(&tmO);
    }
    if (warp == 1) {
        tmem_alloc(misc, Cfg::TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    // ---- union of the tile's selections (warps 2-5) -----------------------
    if (warp >= 2) {
        const int ut = tid - 64;
        for (int i = ut; i < HF_MAX_KEY_BLOCKS / 4; i += 128) sSel[i] = 0;
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const int total = nblk * g.k_eff;
        for (int i = ut; i < total; i += 128) {
            const int gq = i / g.k_eff;
            const int m = i - gq * g.k_eff;
            const int kb = p.idx[((size_t)bh * g.nqb + qb0 + gq) * g.k_eff + m];
            if (kb >= 0 && kb < g.nkb) {
                atomicOr(&sSel[kb >> 2], (1u << gq) << ((kb & 3) * 8));
            } else {
                report_error(wc, HF_DEV_ERR_CHECK, SITE_ATTN_BAD_INDEX);
            }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        // ordered compaction of kb with a non-empty selection mask
        const int w4 = warp - 2;
        int base_out = 0;
        for (int base = 0; base < g.nkb; base += 128) {
            const int kb = base + ut;
            uint32_t m = 0;
            if (kb < g.nkb) m = (sSel[kb >> 2] >> ((kb & 3) * 8)) & 0xFFu;
            const uint32_t ball = __ballot_sync(0xFFFFFFFFu, m != 0);
            if (lane == 0) misc[3 + w4] = __popc(ball);
            asm volatile("bar.sync 1, 128;" ::: "memory");
            int before = base_out;
            for (int q = 0; q < w4; ++q) before += misc[3 + q];
            const int tot = misc[3] + misc[4] + misc[5] + misc[6];
            if (m != 0) sUnion[before + __popc(ball & ((1u << lane) - 1u))] = static_cast<uint32_t>(kb) | (m << 16);
            base_out += tot;
            asm volatile("bar.sync 1, 128;" ::: "memory");
        }
        if (ut == 0) misc[2] = base_out;
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const int nU = static_cast<int>(misc[2]);
    const int n_units = count_units<D, BETA>(sUnion, nU, g.bpf, g.nf);
    const bool bad_input = *wc.abort_flag != 0;

    if (warp == 0) {
        // =================== TMA producer ===================
        if (lane == 0 && !bad_input) {
            bool ok = true;
            mbar_arrive_expect_tx(&bar[B_Q], Cfg::G * Cfg::DCH * BETA * 128);
            for (int gq = 0; gq < Cfg::G; ++gq) {
                const int qb = qb0 + min(gq, nblk - 1);   // missing blocks: reload the last one
                const int c = qb / g.bpf;
                const int j = qb - c * g.bpf;
                for (int m = 0; m < Cfg::DCH; ++m)
                    tma_load_3d(sQ + m * (Cfg::TILE_M * 128) + gq * BETA * 128, &tmQ, &bar[B_Q], 64 * m, j * BETA,
                                bh * g.C + c);
            }
            UnitWalk<D, BETA> walk(sUnion, nU, g.bpf, g.nf);
            int u = 0;
            for (; u < n_units && ok; ++u) {
                const int s = u % Cfg::NS;
                if (u >= Cfg::NS) ok = mbar_wait(&bar[B_KV_EMPTY + s], ((u / Cfg::NS) & 1) ^ 1, wc, SITE_ATTN_KV_EMPTY);
                if (!ok) break;
                Seg seg[2];
                walk.next(seg);
                uint8_t* sK = sStage + s * Cfg::STAGE_BYTES;
                uint8_t* sV = sK + Cfg::KV_BYTES;
                mbar_arrive_expect_tx(&bar[B_KV_FULL + s], Cfg::STAGE_BYTES);
                for (int sg = 0; sg < Cfg::SEGS; ++sg) {
                    const int w = seg[sg].kb / g.bpf;
                    const int plane = bh * g.W + p.sm.s[w];
                    for (int m = 0; m < Cfg::DCH; ++m) {
                        const int off = m * (Cfg::UNIT * 128) + sg * Cfg::SUB * 128;
                        tma_load_3d(sK + off, &tmK, &bar[B_KV_FULL + s], 64 * m, seg[sg].y, plane);
                        tma_load_3d(sV + off, &tmV, &bar[B_KV_FULL + s], 64 * m, seg[sg].y, plane);
                    }
                }
            }
            if (FUSED && ok) {
                // state operands go into the stage buffers once both are free
                for (int v = max(0, n_units - Cfg::NS); v < n_units && ok; ++v)
                    ok = mbar_wait(&bar[B_KV_EMPTY + v % Cfg::NS], (v / Cfg::NS) & 1, wc, SITE_ATTN_KV_EMPTY);
                if (ok) {
                    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.smma) + (size_t)bh * Cfg::LIN_BYTES;
                    mbar_arrive_expect_tx(&bar[B_LIN_FULL], Cfg::LIN_BYTES);
                    bulk_load(sStage, src, Cfg::LIN_BYTES / 2, &bar[B_LIN_FULL]);
                    bulk_load(sStage + Cfg::LIN_BYTES / 2, src + Cfg::LIN_BYTES / 2, Cfg::LIN_BYTES / 2,
                              &bar[B_LIN_FULL]);
                }
            }
            if (!ok) {
                // drain: wait (bounded) for loads already issued
                for (int v = max(0, u - Cfg::NS); v < u; ++v) {
                    const uint32_t a = smem_u32(&bar[B_KV_FULL + v % Cfg::NS]);
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(a, (v / Cfg::NS) & 1) && globaltimer_ns() - t0 < p.wait_limit_ns) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // =================== MMA issuer ===================
        if (lane == 0 && !bad_input) {
            bool ok = mbar_wait(&bar[B_Q], 0, wc, SITE_ATTN_Q);
            tc_fence_after();
            const uint32_t q_base = smem_u32(sQ);
            for (int u = 0; ok && u <= n_units; ++u) {
                if (u < n_units) {
                    const int s = u % Cfg::NS;
                    const int b = u & 1;
                    ok = mbar_wait(&bar[B_KV_FULL + s], (u / Cfg::NS) & 1, wc, SITE_ATTN_KV_FULL);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t k_base = smem_u32(sStage + s * Cfg::STAGE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t qa = q_base + (kk >> 2) * (Cfg::TILE_M * 128) + (kk & 3) * 32;
                        const uint32_t ka = k_base + (kk >> 2) * (Cfg::UNIT * 128) + (kk & 3) * 32;
                        mma_ss(tmem + Cfg::S_COL + b * 64, smem_desc(qa, 16, 1024), smem_desc(ka, 16, 1024),
                               Cfg::IDESC_QK, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&bar[B_S_FULL + b]);
                }
                if (u >= 1) {
                    const int v = u - 1;
                    const int sv = v % Cfg::NS;
                    const int bv = v & 1;
                    ok = mbar_wait(&bar[B_P_FULL + bv], (v >> 1) & 1, wc, SITE_ATTN_P_FULL);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t v_base = smem_u32(sStage + sv * Cfg::STAGE_BYTES + Cfg::KV_BYTES);
#pragma unroll
                    for (int kk = 0; kk < Cfg::UNIT / 16; ++kk) {
                        mma_ts(tmem + Cfg::O_COL, tmem + Cfg::S_COL + bv * 64 + kk * 8,
                               smem_desc(v_base + kk * 2048, Cfg::UNIT * 128, 1024), Cfg::IDESC_PV,
                               (v > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&bar[B_PV_DONE + bv]);
                    mma_commit(&bar[B_KV_EMPTY + sv]);
                }
            }
            if (FUSED && ok) {
                ok = mbar_wait(&bar[B_PHIQ], 0, wc, SITE_ATTN_PHIQ) && mbar_wait(&bar[B_LIN_FULL], 0, wc, SITE_ATTN_LIN);
                if (ok) {
                    tc_fence_after();
                    const uint32_t l_base = smem_u32(sStage);
#pragma unroll
                    for (int hl = 0; hl < 2; ++hl) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t qa = q_base + (kk >> 2) * (Cfg::TILE_M * 128) + (kk & 3) * 32;
                            const uint32_t sa = l_base + hl * (D * D * 2) + kk * 2048;
                            mma_ss(tmem + Cfg::S_COL, smem_desc(qa, 16, 1024), smem_desc(sa, D * 128, 1024),
                                   Cfg::IDESC_LIN, (hl > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(&bar[B_LIN_DONE]);
                }
            }
            // drain: every MMA this thread issued has completed before TMEM is freed
            mma_commit(&bar[B_DRAIN]);
            const uint32_t a = smem_u32(&bar[B_DRAIN]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(a, 0)) {
                if (globaltimer_ns() - t0 > p.wait_limit_ns) {
                    report_error(wc, HF_DEV_ERR_TIMEOUT, SITE_ATTN_DRAIN);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (!bad_input) {
        // =================== softmax / epilogue (warps 2-5) ===================
        const int quarter = warp & 3;            // TMEM lane quarter this warp may access
        const int r = quarter * 32 + lane;       // query row within the tile
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const int gq = min(r / BETA, nblk - 1);  // the row's query block within the tile
        const float sl2 = g.scale_log2;
        float m_run = -INFINITY, m_use = -INFINITY, l = 0.0f;
        bool ok = true;
        UnitWalk<D, BETA> walk(sUnion, nU, g.bpf, g.nf);
        for (int u = 0; u < n_units; ++u) {
            const int b = u & 1;
            Seg seg[2];
            walk.next(seg);
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[B_S_FULL + b], (u >> 1) & 1, wc, SITE_ATTN_S_FULL));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[2][32];
            tmem_ld32(tmem + lane_addr + Cfg::S_COL + b * 64, sr[0]);
            tmem_ld32(tmem + lane_addr + Cfg::S_COL + b * 64 + 32, sr[1]);
            // column validity for this row
            int nv0, nv1;
            if (BETA == 32) {
                nv0 = ((seg[0].sel >> gq) & 1u) ? seg[0].nv : 0;
                nv1 = ((seg[1].sel >> gq) & 1u) ? seg[1].nv : 0;
            } else {
                const int nv = ((seg[0].sel >> gq) & 1u) ? seg[0].nv : 0;
                nv0 = min(nv, 32);
                nv1 = max(0, nv - 32);
            }
            float x[64];
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                x[c] = c < nv0 ? __uint_as_float(sr[0][c]) : -INFINITY;
                x[32 + c] = c < nv1 ? __uint_as_float(sr[1][c]) : -INFINITY;
            }
#pragma unroll
            for (int c = 0; c < 64; ++c) mx = fmaxf(mx, x[c]);
            const float m_new = fmaxf(m_run, mx);
            m_run = m_new;
            // Lazy rescale: the exponent reference m_use only moves when the
            // running max exceeds it by more than 8 (log2 units), so O and l
            // stay consistent with m_use and p <= 2^8.  The TMEM access is
            // warp-collective, so the whole warp enters when any lane needs it.
            const bool move = m_new != -INFINITY && (m_use == -INFINITY || (m_new - m_use) * sl2 > 8.0f);
            const bool scale_o = move && m_use != -INFINITY;   // O already holds earlier units
            if (__any_sync(0xFFFFFFFFu, scale_o)) {
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[B_PV_DONE + ((u - 1) & 1)], ((u - 1) >> 1) & 1, wc,
                                                       SITE_ATTN_PV_DONE));
                if (!ok) break;
                tc_fence_after();
                const float f = scale_o ? ex2_approx((m_use - m_new) * sl2) : 1.0f;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_addr + Cfg::O_COL + c0, o);
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f);
                    tmem_st32(tmem + lane_addr + Cfg::O_COL + c0, o);
                }
                l *= f;
            }
            if (move) m_use = m_new;
            const float neg = (m_use == -INFINITY) ? 0.0f : -m_use * sl2;
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p0 = ex2_approx(fmaf(x[2 * c], sl2, neg));
                const float p1 = ex2_approx(fmaf(x[2 * c + 1], sl2, neg));
                l += p0 + p1;
                pk[c] = pack_bf16(p0, p1);
            }
            tmem_st32(tmem + lane_addr + Cfg::S_COL + b * 64, pk);
            tc_fence_before();
            mbar_arrive(&bar[B_P_FULL + b]);
        }
        if (ok) {
            const int last = n_units - 1;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[B_PV_DONE + (last & 1)], (last >> 1) & 1, wc, SITE_ATTN_PV_DONE));
        }
        const float inv_l = 1.0f / l;
        const int qb = qb0 + gq;
        const int c_frame = qb / g.bpf;
        const int jq = qb - c_frame * g.bpf;
        if (FUSED) {
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
                mbar_arrive(&bar[B_PHIQ]);
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[B_LIN_DONE], 0, wc, SITE_ATTN_LIN));
                if (ok) {
                    tc_fence_after();
                    const float inv_den = 1.0f / den;
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32], li[32];
                        tmem_ld32(tmem + lane_addr + Cfg::O_COL + c0, o);
                        tmem_ld32(tmem + lane_addr + Cfg::S_COL + c0, li);
                        uint8_t* rowp = sQ + (c0 >> 6) * (Cfg::TILE_M * 128) + r * 128;
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch) {
                            uint32_t w4[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int c = ch * 8 + 2 * i;
                                const float a = fmaf(__uint_as_float(o[c]), inv_l, __uint_as_float(li[c]) * inv_den);
                                const float bq =
                                    fmaf(__uint_as_float(o[c + 1]), inv_l, __uint_as_float(li[c + 1]) * inv_den);
                                w4[i] = pack_bf16(a, bq);
                            }
                            const int lch = ((c0 & 63) >> 3) + ch;   // logical 16-byte chunk in the 128-byte row
                            *reinterpret_cast<uint4*>(rowp + (((lch ^ (r & 7)) & 7) << 4)) =
                                make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                    fence_proxy_async_smem();
                }
            }
            if (!ok) *wc.abort_flag = 1;
            // every softmax thread reaches this barrier exactly once
            asm volatile("bar.sync 1, 128;" ::: "memory");
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
            const int rin = r - gq * BETA;
            const bool valid = (r / BETA) < nblk && rin < min(BETA, g.nf - jq * BETA);
            float* dst = p.o_swa + ((size_t)bh * g.C * g.nf + (size_t)c_frame * g.nf + (size_t)jq * BETA + rin) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_addr + Cfg::O_COL + c0, o);
                if (valid) {
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        float4 v4 = make_float4(__uint_as_float(o[c]) * inv_l, __uint_as_float(o[c + 1]) * inv_l,
                                                __uint_as_float(o[c + 2]) * inv_l, __uint_as_float(o[c + 3]) * inv_l);
                        *reinterpret_cast<float4*>(dst + c0 + c) = v4;
                    }
                }
            }
        }
        if (!ok) {
            // keep the MMA thread from waiting on arrivals that will not come
            *wc.abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
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
    kern<<<grid, 192, Cfg::SMEM_ALLOC, st>>>(tq, tk, tv, to, p);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_attn(const uint16_t* Q, const uint16_t* Kc, const uint16_t* Vc, const Geom& g, const SlotMap& sm,
                const int32_t* idx, const uint16_t* smma, const float* z, float* o_swa, uint16_t* o_bf16,
                uint32_t* status, uint64_t wait_limit_ns, void* stream)
{
    const bool fused = o_bf16 != nullptr;
    const int qrows = g.beta;   // Q / O box rows = one query block
    const int kvrows = g.beta < 64 ? g.beta : 64;
    alignas(64) CUtensorMap tq, tk, tv, to;
    int e;
    // Q and O: [BH*C planes][nf rows][d]; K, V: [BH*W slots][nf valid rows][d], slot pitch slot_stride rows
    e = make_tmap_bf16_3d(&tq, Q, g.d, g.nf, (uint64_t)g.BH * g.C, (uint64_t)g.d * 2, (uint64_t)g.nf * g.d * 2, 64,
                          qrows);
    if (e) return e;
    e = make_tmap_bf16_3d(&tk, Kc, g.d, g.nf, (uint64_t)g.BH * g.W, (uint64_t)g.d * 2,
                          (uint64_t)g.slot_stride * g.d * 2, 64, kvrows);
    if (e) return e;
    e = make_tmap_bf16_3d(&tv, Vc, g.d, g.nf, (uint64_t)g.BH * g.W, (uint64_t)g.d * 2,
                          (uint64_t)g.slot_stride * g.d * 2, 64, kvrows);
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
    const int grid = g.BH * p.tiles_per_head;
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
