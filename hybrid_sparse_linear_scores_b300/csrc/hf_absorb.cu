// hf_absorb.cu -- absorption of evicted frames into the linear temporal
// attention state (Hybrid Forcing, English technical summary, section 2.A.1:
// a compact KV state that incrementally aggregates information from evicted
// frames; arXiv abstract: the state "incrementally absorbs evicted tokens"):
//   S[c][j] += sum_t phi(k_t[c]) v_t[j],   z[c] += sum_t phi(k_t[c]).
//
// Per head this is a [d x n] x [n x d] GEMM contracted over the n evicted
// tokens, with about 64 FLOP per byte read: the bound is HBM bandwidth, so the
// design is about keeping every SM streaming.
//
// Work split.  A head's value channels are cut into NG column groups of NV
// channels (NG = d / NV), and each (head, column group) is one thread-block
// cluster of CL CTAs that split the tokens; the host picks NG and CL so that
// all clusters are resident at once (occupancy query) and the CTAs cover the
// SMs.  Every CTA reads all d key channels of its tokens (phi needs them) and
// the NV value channels of its group; a key tile read by both groups of a
// head comes from L2 the second time.
//
// Per 64-token tile: TMA brings the key tile (d channels) and the value tile
// (NV channels) into a stage of a ring of 6-8 stages.  The transform warps compute
// phi(k) for one feature per thread and write it straight into tensor memory
// as the MMA's A operand, as a bf16 pair hi = rn(phi), lo = rn(phi - hi)
// (about 16 significant bits, twice a bf16 operand's); z is summed on the
// way, in float32.  The MMA warp then runs D = phi(K)^T V with A from tensor memory
// and B = the value tile in shared memory (hi and lo: two MMA chains into one
// accumulator), M = 128 features (zero rows when d = 64), N = NV.  The tensor
// core only ever accumulates one tile: two accumulators alternate, and the
// transform warps fold each finished tile into float32 registers with
// round-to-nearest adds while the next one is multiplied.
//
// The CL partial states of a cluster are summed through distributed shared
// memory in rank order and added to S in global memory (no atomics, no
// partial states in HBM): results are deterministic for a given launch shape.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA
// issuer, warps 2-9 phi transform and accumulator folding (feature 32q + lane
// of the warp's TMEM lane quarter q; warps 2-5 take the first 32 tokens of a
// tile and the first half of the accumulator's columns, warps 6-9 the rest).
#include <cooperative_groups.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "hf_internal.h"
#include "hf_ptx.cuh"

namespace cg = cooperative_groups;

namespace hf {
namespace {

constexpr int cmax(int a, int b) { return a > b ? a : b; }

template <int D, int NV, int NSX = 0>
struct AbsCfg {
    static constexpr int TT = 64;                    // tokens per tile
    static constexpr int CHUNK = TT * 128;           // 64 channels x 64 tokens, 128-byte swizzle: 8 KB
    static constexpr int K_BYTES = (D / 64) * CHUNK;
    static constexpr int V_BYTES = (NV / 64) * CHUNK;
    static constexpr int STAGE = K_BYTES + V_BYTES;
    // shared-memory stages (tiles in flight); NSX > 0 chooses fewer, so that the
    // CTA leaves room on its SM for kernels that run beside the absorb
    static constexpr int NS = NSX > 0 ? NSX : (STAGE <= 24 * 1024 ? 8 : 6);
    static constexpr int NA = 4;                     // TMEM A-operand stages
    static constexpr int TW = 16;                    // transform warps: 4 per TMEM lane quarter
    static constexpr int TPW = TT / 4;               // tokens of a tile per transform warp
    static constexpr int NC = NV / 4;                // accumulator columns folded per transform warp
    static constexpr int PITCH = NV + 4;             // partial-state row pitch (floats; rows 16-byte aligned)
    static constexpr int PART_BYTES = 128 * PITCH * 4;
    static constexpr int BUF = cmax(NS * STAGE, PART_BYTES);
    static constexpr int OFF_BAR = BUF;              // mbarriers: FULL[NS], EMPTY[NS], PHI[NA], ACC_FULL[2], ACC_FREE[2], DRAIN
    static constexpr int NBAR = 2 * NS + NA + 5;
    static constexpr int OFF_MISC = OFF_BAR + 8 * 32;             // uint32 [16]
    static constexpr int OFF_ZP = OFF_MISC + 64;                  // fp32 [4][128] z partials (token quarters)
    static constexpr int SMEM = OFF_ZP + 4 * 128 * 4;
    // more than half of an SM's shared memory: one CTA per SM, so that its
    // 512 TMEM columns are always free when it starts
    static constexpr int SMEM_ALLOC = cmax(SMEM + 1024, 116 * 1024);
    static constexpr uint32_t A_COLS = 64;           // per A stage: hi [0, 32), lo [32, 64)
    static constexpr uint32_t ACC0 = NA * A_COLS;    // accumulators at ACC0 + b * NV
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(ACC0 + 2 * NV <= TMEM_COLS, "TMEM budget");
    static_assert(NBAR <= 32, "barrier slots");
    static_assert(NS >= NA, "a TMEM stage is rewritten only after its MMA completed");
    static constexpr uint32_t IDESC = idesc_bf16_f32(128, NV, false, true);   // A from TMEM, B MN-major
    static constexpr int NTHR = 32 * (2 + TW);
    static constexpr int B_FULL = 0, B_EMPTY = NS, B_PHI = 2 * NS, B_ACC_FULL = 2 * NS + NA,
                         B_ACC_FREE = B_ACC_FULL + 2, B_DRAIN = B_ACC_FREE + 2;
};

// misc words
enum { X_TMEM = 0, X_ABORT = 1 };

struct AbsParams {
    int BH, n, NG, CL;
    float* S;
    float* z;
    uint32_t* status;
    uint64_t wait_limit_ns;
    uint16_t* smma;   // optional: the new S also as the linear read's bf16 hi/lo MMA operand
};

template <int D, int NV, int NSX = 0>
__global__ void __launch_bounds__(AbsCfg<D, NV, NSX>::NTHR, 1)
    absorb_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const AbsParams p)
{
    using Cfg = AbsCfg<D, NV, NSX>;
    constexpr int NS = Cfg::NS, NA = Cfg::NA;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
    float* zp = reinterpret_cast<float*>(smem + Cfg::OFF_ZP);

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int cid = blockIdx.x / p.CL;                 // cluster = (head, column group)
    const int bh = cid / p.NG;
    const int grp = cid - bh * p.NG;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_tiles = (p.n + Cfg::TT - 1) / Cfg::TT;
    const int t_begin = (int)((long)rank * n_tiles / p.CL);
    const int t_end = (int)((long)(rank + 1) * n_tiles / p.CL);
    const int my_tiles = t_end - t_begin;

    WaitCtl wc{reinterpret_cast<volatile uint32_t*>(misc + X_ABORT), p.status, p.wait_limit_ns};

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar[Cfg::B_FULL + s], 1);
            mbar_init(&bar[Cfg::B_EMPTY + s], 1);
        }
        for (int s = 0; s < NA; ++s) mbar_init(&bar[Cfg::B_PHI + s], 32 * Cfg::TW);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bar[Cfg::B_ACC_FULL + b], 1);
            mbar_init(&bar[Cfg::B_ACC_FREE + b], 32 * Cfg::TW);
        }
        mbar_init(&bar[Cfg::B_DRAIN], 1);
        misc[X_ABORT] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(misc + X_TMEM, Cfg::TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[X_TMEM];

    // this CTA's rows of the state slice it updates, read up front by the
    // transform warps (idle until the first tile lands; their latency hides
    // behind the token stream)
    const int rows_per = (D + p.CL - 1) / p.CL;
    const int r0 = min(D, rank * rows_per), r1 = min(D, r0 + rows_per);
    constexpr int C4 = NV / 4;                          // float4 per row of the slice
    constexpr int PRE = 4;                              // float4 items prefetched per transform thread
    constexpr int NT = 32 * Cfg::TW;                    // transform threads
    const int tt = tid - 64;                            // transform thread index (< 0 for warps 0, 1)
    float* Sg = p.S + (size_t)bh * D * D + grp * NV;
    float4 s_old[PRE];
    if (tt >= 0) {
#pragma unroll
        for (int it = 0; it < PRE; ++it) {
            const int e = tt + it * NT;
            if (e < (r1 - r0) * C4)
                s_old[it] = *reinterpret_cast<const float4*>(Sg + (size_t)(r0 + e / C4) * D + 4 * (e % C4));
        }
    }

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            bool ok = true;
            int i = 0;
            for (; i < my_tiles && ok; ++i) {
                const int s = i % NS;
                if (i >= NS) ok = mbar_wait(&bar[Cfg::B_EMPTY + s], ((i / NS) - 1) & 1, wc, SITE_ABSORB_EMPTY);
                if (!ok) break;
                uint8_t* st = smem + s * Cfg::STAGE;
                const int row = (t_begin + i) * Cfg::TT;
                mbar_arrive_expect_tx(&bar[Cfg::B_FULL + s], Cfg::STAGE);
                for (int m = 0; m < D / 64; ++m)
                    tma_load_3d(st + m * Cfg::CHUNK, &tmK, &bar[Cfg::B_FULL + s], 64 * m, row, bh);
                for (int m = 0; m < NV / 64; ++m)
                    tma_load_3d(st + Cfg::K_BYTES + m * Cfg::CHUNK, &tmV, &bar[Cfg::B_FULL + s], grp * NV + 64 * m,
                                row, bh);
            }
            // bounded drain: every load issued has landed before the CTA goes on
            for (int v = (i > NS ? i - NS : 0); v < i; ++v) {
                const uint32_t a = smem_u32(&bar[Cfg::B_FULL + v % NS]);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(a, (v / NS) & 1) && globaltimer_ns() - t0 < p.wait_limit_ns) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            bool ok = true;
            for (int i = 0; i < my_tiles && ok; ++i) {
                const int s = i % NS, as = i % NA, a = i & 1;
                ok = mbar_wait(&bar[Cfg::B_PHI + as], (i / NA) & 1, wc, SITE_ABSORB_PHI);
                if (ok && i >= 2) ok = mbar_wait(&bar[Cfg::B_ACC_FREE + a], ((i >> 1) - 1) & 1, wc, SITE_ABSORB_ACC);
                if (!ok) break;
                tc_fence_after();
                const uint64_t vdesc = smem_desc(smem_u32(smem + s * Cfg::STAGE + Cfg::K_BYTES), Cfg::CHUNK, 1024);
                const uint32_t acc = tmem + Cfg::ACC0 + a * NV;
                const uint32_t at = tmem + as * Cfg::A_COLS;
#pragma unroll
                for (int hl = 0; hl < 2; ++hl) {
#pragma unroll
                    for (int kk = 0; kk < Cfg::TT / 16; ++kk)
                        mma_ts(acc, at + 32 * hl + 8 * kk, vdesc + (uint64_t)((kk * 2048) >> 4), Cfg::IDESC,
                               (hl > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bar[Cfg::B_EMPTY + s]);
                mma_commit(&bar[Cfg::B_ACC_FULL + a]);
            }
            // drain (bounded): every MMA issued has completed
            mma_commit(&bar[Cfg::B_DRAIN]);
            const uint32_t a = smem_u32(&bar[Cfg::B_DRAIN]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(a, 0)) {
                if (globaltimer_ns() - t0 > p.wait_limit_ns) {
                    report_error(wc, HF_DEV_ERR_TIMEOUT, SITE_ABSORB_DRAIN);
                    break;
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- phi transform + accumulator folding ----------------
        const int q = warp & 3;                  // TMEM lane quarter
        const int tq = (warp - 2) >> 2;          // token quarter of a tile, column quarter of the accumulator
        const int f = 32 * q + lane;             // feature (TMEM lane)
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        constexpr int NC = Cfg::NC;
        const uint8_t* kcol0 = smem + (uint32_t)(f / 64) * Cfg::CHUNK;
        float racc[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) racc[k] = 0.0f;
        float z_run = 0.0f;
        bool ok = true;
        auto fold = [&](int j) -> bool {
            const int a = j & 1;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar[Cfg::B_ACC_FULL + a], (j >> 1) & 1, wc, SITE_ABSORB_ACC)))
                return false;
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < NC; c0 += 16) {
                uint32_t v[16];
                tmem_ld16_nw(tmem + lane_base + Cfg::ACC0 + a * NV + tq * NC + c0, v);
                tmem_wait_ld();
                reg_dep16(v);
#pragma unroll
                for (int k = 0; k < 16; ++k) racc[c0 + k] = __fadd_rn(racc[c0 + k], __uint_as_float(v[k]));
            }
            tc_fence_before();
            mbar_arrive(&bar[Cfg::B_ACC_FREE + a]);
            return true;
        };
        constexpr float kLog2e = 1.4426950408889634f;
        for (int i = 0; i < my_tiles && ok; ++i) {
            const int s = i % NS, as = i % NA;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[Cfg::B_FULL + s], (i / NS) & 1, wc, SITE_ABSORB_FULL));
            if (!ok) break;
            const uint8_t* kt = kcol0 + s * Cfg::STAGE;
            const int tok0 = (t_begin + i) * Cfg::TT + Cfg::TPW * tq;   // first token of this warp's quarter tile
            const bool full = (t_begin + i + 1) * Cfg::TT <= p.n;
            // the quarter tile's keys of feature f (bf16 -> fp32 is a shift)
            float xk[Cfg::TPW];
#pragma unroll
            for (int t = 0; t < Cfg::TPW; ++t) {
                uint32_t h16 = 0;
                if (f < D)
                    h16 = *reinterpret_cast<const uint16_t*>(kt + sw128_offset(Cfg::TPW * tq + t, (uint32_t)(f % 64)));
                xk[t] = __uint_as_float(h16 << 16);
            }
            // phi(x) = max(x, 0) + exp(min(x, 0)) (= elu(x) + 1), two tokens per
            // step; hi = rn(phi), lo = rn(phi - hi)
            uint32_t hi[Cfg::TPW / 2], lo[Cfg::TPW / 2];
            float za = 0.0f, zb = 0.0f;   // this quarter tile's even / odd tokens: short chains
#pragma unroll
            for (int j = 0; j < Cfg::TPW / 2; ++j) {
                const float xa = xk[2 * j], xb = xk[2 * j + 1];
                float ea, eb;
                mul2(ea, eb, fminf(xa, 0.0f), fminf(xb, 0.0f), kLog2e, kLog2e);
                ea = ex2_approx(ea);
                eb = ex2_approx(eb);
                float ya, yb;
                add2(ya, yb, fmaxf(xa, 0.0f), fmaxf(xb, 0.0f), ea, eb);
                if (!full) {   // tokens past the last evicted one (and features past d) carry phi = 0
                    ya = (f < D && tok0 + 2 * j < p.n) ? ya : 0.0f;
                    yb = (f < D && tok0 + 2 * j + 1 < p.n) ? yb : 0.0f;
                } else if (f >= D) {
                    ya = yb = 0.0f;
                }
                add2(za, zb, za, zb, ya, yb);
                const uint32_t h = pack_bf16(ya, yb);
                hi[j] = h;
                float ra, rb;   // phi - hi, with -hi taken from the packed bits (sign flipped)
                add2(ra, rb, ya, yb, __uint_as_float((h << 16) ^ 0x80000000u),
                     __uint_as_float((h & 0xFFFF0000u) ^ 0x80000000u));
                lo[j] = pack_bf16(ra, rb);
            }
            z_run += za + zb;
            const uint32_t at = tmem + lane_base + as * Cfg::A_COLS + (Cfg::TPW / 2) * tq;
            tmem_st8_nw(at, hi);
            tmem_st8_nw(at + 32, lo);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bar[Cfg::B_PHI + as]);
            if (i >= 1) ok = fold(i - 1);
        }
        if (ok && my_tiles > 0) ok = fold(my_tiles - 1);
        // every load was consumed and the last MMA has completed (its
        // accumulator was folded), so the stage buffers are free: partial
        // state [128][PITCH] over them
        float* part = reinterpret_cast<float*>(smem);
        if (ok) {
#pragma unroll
            for (int k = 0; k < NC; k += 4)
                *reinterpret_cast<float4*>(part + f * Cfg::PITCH + tq * NC + k) =
                    make_float4(racc[k], racc[k + 1], racc[k + 2], racc[k + 3]);
            zp[tq * 128 + f] = z_run;
        } else {
            *wc.abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster.sync();
    // ---- cluster reduction: rank r owns rows [r0, r1) of this group's columns ----
    // (a CTA that gave up has recorded the error; the state is then undefined)
    if (*wc.abort_flag == 0) {
        auto reduce_item = [&](int e, float4 old) {
            const int c = r0 + e / C4, j = 4 * (e % C4);
            float4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < p.CL)
                    v[q] = *reinterpret_cast<const float4*>(
                        cluster.map_shared_rank(reinterpret_cast<float*>(smem), q) + c * Cfg::PITCH + j);
            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (q < p.CL) {
                    acc.x += v[q].x;
                    acc.y += v[q].y;
                    acc.z += v[q].z;
                    acc.w += v[q].w;
                }
            }
            const float4 nv = make_float4(old.x + acc.x, old.y + acc.y, old.z + acc.z, old.w + acc.w);
            *reinterpret_cast<float4*>(Sg + (size_t)c * D + j) = nv;
            if (p.smma != nullptr) {
                // hi = rn(S), lo = rn(S - hi), MN-major with the 128-byte swizzle:
                // per head [hi | lo][column / 64][row c][128 B], 16-byte chunks of
                // 8 columns XOR-ed with (c mod 8); these 4 columns are one half chunk
                const int jj = grp * NV + j;   // column of the head's state
                const uint32_t h0 = pack_bf16(nv.x, nv.y), h1 = pack_bf16(nv.z, nv.w);
                const uint32_t l0 = pack_bf16(nv.x - bf16_lo(h0), nv.y - bf16_hi(h0));
                const uint32_t l1 = pack_bf16(nv.z - bf16_lo(h1), nv.w - bf16_hi(h1));
                const uint32_t off = (uint32_t)(jj / 64) * (uint32_t)(D * 128) + (uint32_t)c * 128u +
                                     (((((uint32_t)jj % 64u) >> 3) ^ ((uint32_t)c & 7u)) << 4) + ((uint32_t)jj & 4u) * 2u;
                uint8_t* base = reinterpret_cast<uint8_t*>(p.smma) + (size_t)bh * 2 * D * D * 2;
                *reinterpret_cast<uint2*>(base + off) = make_uint2(h0, h1);
                *reinterpret_cast<uint2*>(base + (size_t)D * D * 2 + off) = make_uint2(l0, l1);
            }
        };
        const int total = (r1 - r0) * C4;
        if (tt >= 0) {
#pragma unroll
            for (int it = 0; it < PRE; ++it) {
                const int e = tt + it * NT;
                if (e < total) reduce_item(e, s_old[it]);
            }
            for (int e = tt + PRE * NT; e < total; e += NT)
                reduce_item(e, *reinterpret_cast<const float4*>(Sg + (size_t)(r0 + e / C4) * D + 4 * (e % C4)));
        } else if (grp == 0 && rank == 0) {
            // z: warps 0 and 1, one feature per thread (rows d..127 of the
            // d = 64 case are zero); every rank's four partials requested first
            for (int c = tid; c < D; c += 64) {
                float4 zv[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (q < p.CL) {
                        const float* zq = cluster.map_shared_rank(zp, q);
                        zv[q] = make_float4(zq[c], zq[128 + c], zq[256 + c], zq[384 + c]);
                    }
                }
                float acc = 0.0f;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q < p.CL) acc += (zv[q].x + zv[q].y) + (zv[q].z + zv[q].w);
                p.z[(size_t)bh * D + c] += acc;
            }
        }
    }
    cluster.sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

template <int D, int NV, int NSX = 0>
cudaLaunchConfig_t absorb_launch_cfg(int grid, int CL, cudaStream_t st, cudaLaunchAttribute* attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(AbsCfg<D, NV, NSX>::NTHR);
    cfg.dynamicSmemBytes = AbsCfg<D, NV, NSX>::SMEM_ALLOC;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Clusters of CL CTAs of absorb_kernel<D, NV, NSX> that fit on the device at
// once (cached per device; 0 if the query fails).
template <int D, int NV, int NSX = 0>
int max_clusters(int dev, int CL)
{
    static std::mutex mu;
    static int cache[64][9] = {};
    if (dev < 0 || dev >= 64 || CL < 1 || CL > 8) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev][CL] == 0) {
        auto kern = absorb_kernel<D, NV, NSX>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, AbsCfg<D, NV, NSX>::SMEM_ALLOC) !=
            cudaSuccess)
            return 0;
        cudaLaunchAttribute attr[1];
        const cudaLaunchConfig_t cfg = absorb_launch_cfg<D, NV, NSX>(CL, CL, 0, attr);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            return 0;
        }
        cache[dev][CL] = n;
    }
    return cache[dev][CL];
}

template <int D, int NV, int NSX = 0>
int launch_absorb_t(const CUtensorMap& tk, const CUtensorMap& tv, AbsParams p, cudaStream_t st)
{
    using Cfg = AbsCfg<D, NV, NSX>;
    auto kern = absorb_kernel<D, NV, NSX>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC);
    if (e != cudaSuccess) return (int)e;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = absorb_launch_cfg<D, NV, NSX>(p.BH * p.NG * p.CL, p.CL, st, attr);
    e = cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

// The launch shape: NG column groups per head and CL CTAs per cluster, the
// most CTAs (counted up to one per SM) whose clusters are all resident at
// once; on ties, the larger cluster, and fewer column groups (fewer repeated
// key reads).  Clusters of one CTA never wait on each other, so they may run
// in several waves.
template <int D, int NV, int NSX = 0>
void pick_shape(int BH, int n_tiles, int sms, int dev, int NG, int& best_cl, int& best_score)
{
    // sharing the SMs (NSX > 0): at most half of them
    const int max_cl = NSX > 0 ? 6 : 8;
    if (NSX > 0) sms = (sms + 1) / 2;
    for (int CL = max_cl; CL >= 1; --CL) {
        if (CL > n_tiles && CL > 1) continue;
        const long clusters = (long)BH * NG;
        const long ctas = clusters * CL;
        if (CL > 1 && (ctas > sms || clusters > max_clusters<D, NV, NSX>(dev, CL))) continue;
        const int score = (int)(ctas < sms ? ctas : sms);
        if (score > best_score) {
            best_score = score;
            best_cl = CL;
        }
    }
}


// The shape and the launch, for one stage count (NSX: 0 = the default).
template <int NSX>
int launch_absorb_ns(const CUtensorMap& tk, const CUtensorMap& tv, const Geom& g, AbsParams p, int n_tiles, int sms,
                     int dev, cudaStream_t st)
{
    if (g.d == 64) {
        int cl = 1, ctas = 0;
        pick_shape<64, 64, NSX>(g.BH, n_tiles, sms, dev, 1, cl, ctas);
        p.CL = cl;
        return launch_absorb_t<64, 64, NSX>(tk, tv, p, st);
    }
    int cl1 = 1, c1 = 0, cl2 = 1, c2 = 0;
    pick_shape<128, 128, NSX>(g.BH, n_tiles, sms, dev, 1, cl1, c1);
    pick_shape<128, 64, NSX>(g.BH, n_tiles, sms, dev, 2, cl2, c2);
    // two column groups compute phi of every key twice: worth it only for
    // clearly more CTAs
    if (2 * c2 > 3 * c1) {
        p.NG = 2;
        p.CL = cl2;
        return launch_absorb_t<128, 64, NSX>(tk, tv, p, st);
    }
    p.CL = cl1;
    return launch_absorb_t<128, 128, NSX>(tk, tv, p, st);
}

}  // namespace

int launch_absorb(const uint16_t* K_ev, const uint16_t* V_ev, int32_t n_ev, int64_t head_stride, const Geom& g,
                  float* S, float* z, uint16_t* smma, bool share_sms, uint32_t* status, uint64_t wait_limit_ns,
                  void* stream)
{
    alignas(64) CUtensorMap tk, tv;
    const uint64_t hs = (uint64_t)head_stride * g.d * 2;
    constexpr int TT = AbsCfg<128, 64>::TT;
    int e = make_tmap_bf16_3d(&tk, K_ev, g.d, (uint64_t)n_ev, g.BH, (uint64_t)g.d * 2, hs, 64, TT);
    if (e) return e;
    e = make_tmap_bf16_3d(&tv, V_ev, g.d, (uint64_t)n_ev, g.BH, (uint64_t)g.d * 2, hs, 64, TT);
    if (e) return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int n_tiles = (n_ev + TT - 1) / TT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    AbsParams p{g.BH, n_ev, 1, 1, S, z, status, wait_limit_ns, smma};
    // sharing: clusters of at most 6 CTAs on about half of the SMs, four
    // stages (about 130 KB of shared memory instead of 193), so that the key
    // pooling and the forward's prologue fit beside the absorb
    return share_sms ? launch_absorb_ns<4>(tk, tv, g, p, n_tiles, sms, dev, st)
                     : launch_absorb_ns<0>(tk, tv, g, p, n_tiles, sms, dev, st);
}

}  // namespace hf
