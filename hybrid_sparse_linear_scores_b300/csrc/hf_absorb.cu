// hf_absorb.cu -- absorption of evicted frames into the linear temporal
// attention state (Hybrid Forcing, English technical summary, section 2.A.1:
// a compact KV state that incrementally aggregates information from evicted
// frames; arXiv abstract: the state "incrementally absorbs evicted tokens"):
//   S[c][j] += sum_t phi(k_t[c]) v_t[j],   z[c] += sum_t phi(k_t[c]).
//
// Per head this is a [d x n] x [n x d] GEMM contracted over the n evicted
// tokens: tcgen05 with M = 128 (phi features; zero-padded when d = 64),
// N = d (value channels), both operands MN-major straight from the TMA tiles.
// phi(k) enters the MMA as a bf16 pair hi + lo (hi = rn(phi), lo =
// rn(phi - hi)), two MMAs into one fp32 accumulator, so S keeps ~16 bits
// more than a bf16 operand would give; z is summed in fp32 on CUDA cores.
// The tensor-core accumulator only ever holds one 64-token tile: two TMEM
// accumulators alternate, and the epilogue warps fold each finished tile
// into fp32 registers with round-to-nearest adds while the next tile is
// multiplied, so long absorbs do not accumulate the tensor core's internal
// rounding over thousands of steps.
//
// One thread-block cluster (CL <= 8 CTAs) per head splits the tokens; the
// CL partial states are summed through distributed shared memory in rank
// order, then added to S in global memory: deterministic, no atomics, no
// partial states in HBM.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA
// issuer, warps 2-9 phi transform (in place over the K tile) and epilogue.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "hf_internal.h"
#include "hf_ptx.cuh"

namespace cg = cooperative_groups;

namespace hf {
namespace {

template <int D>
struct AbsCfg {
    static constexpr int TT = 64;                    // tokens per tile (MMA K extent per tile)
    static constexpr int NS = 4;                     // stages
    static constexpr int CHUNK = TT * 128;           // one 64-column chunk of a tile: 8 KB
    static constexpr int OFF_K = 0;                  // 2 chunks (chunk 1 zero when D = 64)
    static constexpr int OFF_LO = 2 * CHUNK;         // 2 chunks
    static constexpr int OFF_V = 4 * CHUNK;          // D/64 chunks
    static constexpr int STAGE = OFF_V + (D / 64) * CHUNK;
    static constexpr int OFF_MISC = NS * STAGE;
    static constexpr int NBAR = 20;
    static_assert(NS <= 4, "barrier slots hold at most 4 stages");
    static constexpr int OFF_ZP = OFF_MISC + 64 + 8 * NBAR;   // fp32 [8][D] z partials
    static constexpr uint32_t TMEM_COLS = 256;                 // two accumulators of 128 columns
    static constexpr int SMEM = OFF_ZP + 8 * D * 4;
    static constexpr int SMEM_ALLOC = SMEM + 1024;
    static constexpr int PITCH = D + 4;              // partial-state row pitch (floats; rows 16-byte aligned)
    static_assert(128 * PITCH * 4 <= NS * STAGE, "partial state must fit in the stage buffers");
    static constexpr uint32_t IDESC = idesc_bf16_f32(128, D, true, true);
    static constexpr int NTHR = 320;
};

// barrier slots: A_FULL, A_PHI, A_EMPTY have one per stage (NS <= 4)
enum { A_FULL = 0, A_PHI = 4, A_EMPTY = 8, A_ACC_FULL = 12, A_ACC_FREE = 14, A_DRAIN = 16 };

struct AbsParams {
    int BH, n, CL;
    float* S;
    float* z;
    uint32_t* status;
    uint64_t wait_limit_ns;
};

template <int D>
__global__ void __launch_bounds__(320, 1)
    absorb_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const AbsParams p)
{
    using Cfg = AbsCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);      // [0] tmem, [1] abort
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_MISC + 64);
    float* zp = reinterpret_cast<float*>(smem + Cfg::OFF_ZP);

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int bh = blockIdx.x / p.CL;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_tiles = (p.n + Cfg::TT - 1) / Cfg::TT;
    const int t_begin = (int)((long)rank * n_tiles / p.CL);
    const int t_end = (int)((long)(rank + 1) * n_tiles / p.CL);
    const int my_tiles = t_end - t_begin;

    WaitCtl wc{reinterpret_cast<volatile uint32_t*>(misc + 1), p.status, p.wait_limit_ns};

    if (tid == 0) {
        for (int s = 0; s < Cfg::NS; ++s) {
            mbar_init(&bar[A_FULL + s], 1);
            mbar_init(&bar[A_PHI + s], 256);
            mbar_init(&bar[A_EMPTY + s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bar[A_ACC_FULL + b], 1);
            mbar_init(&bar[A_ACC_FREE + b], 256);
        }
        mbar_init(&bar[A_DRAIN], 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    if (D == 64) {   // the zero halves of the M = 128 operands
        for (int s = 0; s < Cfg::NS; ++s)
            for (int i = tid; i < Cfg::CHUNK / 16; i += Cfg::NTHR) {
                reinterpret_cast<uint4*>(smem + s * Cfg::STAGE + Cfg::OFF_K + Cfg::CHUNK)[i] = make_uint4(0, 0, 0, 0);
                reinterpret_cast<uint4*>(smem + s * Cfg::STAGE + Cfg::OFF_LO + Cfg::CHUNK)[i] = make_uint4(0, 0, 0, 0);
            }
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(misc, Cfg::TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            bool ok = true;
            int i = 0;
            for (; i < my_tiles && ok; ++i) {
                const int s = i % Cfg::NS;
                if (i >= Cfg::NS) ok = mbar_wait(&bar[A_EMPTY + s], ((i / Cfg::NS) & 1) ^ 1, wc, SITE_ABSORB_EMPTY);
                if (!ok) break;
                uint8_t* st = smem + s * Cfg::STAGE;
                const int row = (t_begin + i) * Cfg::TT;
                mbar_arrive_expect_tx(&bar[A_FULL + s], 2 * Cfg::TT * D * 2);
                for (int m = 0; m < D / 64; ++m) {
                    tma_load_3d(st + Cfg::OFF_K + m * Cfg::CHUNK, &tmK, &bar[A_FULL + s], 64 * m, row, bh);
                    tma_load_3d(st + Cfg::OFF_V + m * Cfg::CHUNK, &tmV, &bar[A_FULL + s], 64 * m, row, bh);
                }
            }
            if (!ok) {
                for (int v = max(0, i - Cfg::NS); v < i; ++v) {
                    const uint32_t a = smem_u32(&bar[A_FULL + v % Cfg::NS]);
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(a, (v / Cfg::NS) & 1) && globaltimer_ns() - t0 < p.wait_limit_ns) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            for (int i = 0; i < my_tiles && ok; ++i) {
                const int s = i % Cfg::NS;
                const int a = i & 1;
                ok = mbar_wait(&bar[A_PHI + s], (i / Cfg::NS) & 1, wc, SITE_ABSORB_PHI);
                if (ok && i >= 2) ok = mbar_wait(&bar[A_ACC_FREE + a], ((i >> 1) & 1) ^ 1, wc, SITE_ABSORB_ACC);
                if (!ok) break;
                tc_fence_after();
                const uint32_t st = smem_u32(smem + s * Cfg::STAGE);
#pragma unroll
                for (int hl = 0; hl < 2; ++hl) {
                    const uint32_t a0 = st + (hl ? Cfg::OFF_LO : Cfg::OFF_K);
#pragma unroll
                    for (int kk = 0; kk < Cfg::TT / 16; ++kk) {
                        mma_ss(tmem + a * 128, smem_desc(a0 + kk * 2048, Cfg::CHUNK, 1024),
                               smem_desc(st + Cfg::OFF_V + kk * 2048, Cfg::CHUNK, 1024), Cfg::IDESC,
                               (hl > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                mma_commit(&bar[A_EMPTY + s]);
                mma_commit(&bar[A_ACC_FULL + a]);
            }
            mma_commit(&bar[A_DRAIN]);
            const uint32_t a = smem_u32(&bar[A_DRAIN]);
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
        // ---- phi transform: thread -> column pair cp, row group rg ----------
        const int t = tid - 64;                 // 0..255
        constexpr int NCP = D / 2;              // column pairs
        constexpr int NRG = 256 / NCP;          // row groups (4 for d=128, 8 for d=64)
        const int cp = t % NCP, rg = t / NCP;
        const int col = 2 * cp;
        const uint32_t coff = (uint32_t)(col / 64) * Cfg::CHUNK;
        // accumulator drain: warp -> TMEM lane quarter, column half
        constexpr int DC = D / 2;               // columns per draining thread
        const int quarter = warp & 3;
        const int chalf = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        float racc[DC];
#pragma unroll
        for (int k = 0; k < DC; ++k) racc[k] = 0.0f;
        float z0 = 0.0f, z1 = 0.0f;
        bool ok = true;
        auto drain = [&](int j) -> bool {
            const int a = j & 1;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar[A_ACC_FULL + a], (j >> 1) & 1, wc, SITE_ABSORB_ACC)))
                return false;
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < DC; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + a * 128 + chalf * DC + c0, v);
#pragma unroll
                for (int k = 0; k < 32; ++k) racc[c0 + k] = __fadd_rn(racc[c0 + k], __uint_as_float(v[k]));
            }
            tc_fence_before();
            mbar_arrive(&bar[A_ACC_FREE + a]);
            return true;
        };
        for (int i = 0; i < my_tiles && ok; ++i) {
            const int s = i % Cfg::NS;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[A_FULL + s], (i / Cfg::NS) & 1, wc, SITE_ABSORB_FULL));
            if (!ok) break;
            uint8_t* st = smem + s * Cfg::STAGE;
            const int tok0 = (t_begin + i) * Cfg::TT;
            // all rows are loaded before any is written back (the in-place stores
            // could otherwise alias the next row's load, serializing the rows);
            // rows past the last token (a partial tile) become phi = 0
            constexpr int RPT = Cfg::TT / NRG;   // rows per thread
            uint32_t kv[RPT];
#pragma unroll
            for (int k = 0; k < RPT; ++k)
                kv[k] = *reinterpret_cast<const uint32_t*>(st + Cfg::OFF_K + coff + sw128_offset(rg + k * NRG, col % 64));
#pragma unroll
            for (int k = 0; k < RPT; ++k) {
                const int r = rg + k * NRG;
                const bool valid = tok0 + r < p.n;
                float a = bf16_lo(kv[k]), b = bf16_hi(kv[k]);
                a = a > 0.0f ? a + 1.0f : __expf(a);
                b = b > 0.0f ? b + 1.0f : __expf(b);
                a = valid ? a : 0.0f;
                b = valid ? b : 0.0f;
                z0 += a;
                z1 += b;
                const uint32_t hi = pack_bf16(a, b);
                const uint32_t off = coff + sw128_offset(r, col % 64);
                *reinterpret_cast<uint32_t*>(st + Cfg::OFF_K + off) = hi;
                *reinterpret_cast<uint32_t*>(st + Cfg::OFF_LO + off) = pack_bf16(a - bf16_lo(hi), b - bf16_hi(hi));
            }
            fence_proxy_async_smem();
            mbar_arrive(&bar[A_PHI + s]);
            if (i >= 1) ok = drain(i - 1);
        }
        if (ok && my_tiles > 0) ok = drain(my_tiles - 1);
        zp[rg * D + col] = z0;
        zp[rg * D + col + 1] = z1;
        // ---- partial state -> shared memory (over stage 0) ----------------
        __syncwarp();
        float* part = reinterpret_cast<float*>(smem);   // [128][PITCH], over the stage buffers
        // every load was consumed above, and the last MMA has been drained.
        if (ok) {
#pragma unroll
            for (int k = 0; k < DC; k += 4)
                *reinterpret_cast<float4*>(part + row * Cfg::PITCH + chalf * DC + k) =
                    make_float4(racc[k], racc[k + 1], racc[k + 2], racc[k + 3]);
        } else {
            *wc.abort_flag = 1;
        }
    }
    // this rank's rows of S, read while the other CTAs of the cluster finish
    const int rows_per = (D + p.CL - 1) / p.CL;
    const int r0 = rank * rows_per, r1 = min(D, r0 + rows_per);
    float* Sg = p.S + (size_t)bh * D * D;
    constexpr int ITEMS = (D / 8) * (D / 4) / Cfg::NTHR + 1;   // float4 items per thread (rows_per <= D/8 for CL = 8)
    float4 s_old[ITEMS];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int e = tid + it * Cfg::NTHR;
        if (e < (r1 - r0) * (D / 4))
            s_old[it] = *reinterpret_cast<const float4*>(Sg + (size_t)(r0 + e / (D / 4)) * D + 4 * (e % (D / 4)));
    }
    tc_fence_before();
    __syncthreads();
    // z partial of this CTA: fixed order over row groups
    if (tid < D) {
        constexpr int NRG = 256 / (D / 2);
        float acc = 0.0f;
        for (int g2 = 0; g2 < NRG; ++g2) acc += zp[g2 * D + tid];
        zp[7 * D + tid] = acc;   // slot 7 (>= NRG for d=128; for d=64 read after the sum)
    }
    cluster.sync();
    // ---- cluster reduction: rank r owns rows [r0, r1) of S ----------------
    if (*wc.abort_flag == 0) {
        // all ranks' float4s of an item are requested first, then added in rank order;
        // the first ITEMS items of a thread use the prefetched S, any further ones
        // (clusters smaller than 8) read S here
        const int total = (r1 - r0) * (D / 4);
        auto reduce_item = [&](int e, float4 o) {
            const int c = r0 + e / (D / 4), j = 4 * (e % (D / 4));
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
            o.x += acc.x;
            o.y += acc.y;
            o.z += acc.z;
            o.w += acc.w;
            *reinterpret_cast<float4*>(Sg + (size_t)c * D + j) = o;
        };
#pragma unroll
        for (int it = 0; it < ITEMS; ++it) {
            const int e = tid + it * Cfg::NTHR;
            if (e < total) reduce_item(e, s_old[it]);
        }
        for (int e = tid + ITEMS * Cfg::NTHR; e < total; e += Cfg::NTHR)
            reduce_item(e, *reinterpret_cast<const float4*>(Sg + (size_t)(r0 + e / (D / 4)) * D + 4 * (e % (D / 4))));
        if (rank == 0 && tid < D) {
            float acc = 0.0f;
            for (int q = 0; q < p.CL; ++q) acc += cluster.map_shared_rank(zp, q)[7 * D + tid];
            p.z[(size_t)bh * D + tid] += acc;
        }
    }
    cluster.sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

template <int D>
int launch_absorb_t(const CUtensorMap& tk, const CUtensorMap& tv, const AbsParams& p, cudaStream_t st)
{
    using Cfg = AbsCfg<D>;
    auto kern = absorb_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC);
    if (e != cudaSuccess) return (int)e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.BH * p.CL);
    cfg.blockDim = dim3(Cfg::NTHR);
    cfg.dynamicSmemBytes = Cfg::SMEM_ALLOC;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

}  // namespace

int launch_absorb(const uint16_t* K_ev, const uint16_t* V_ev, int32_t n_ev, int64_t head_stride, const Geom& g,
                  float* S, float* z, uint32_t* status, uint64_t wait_limit_ns, void* stream)
{
    alignas(64) CUtensorMap tk, tv;
    const uint64_t hs = (uint64_t)head_stride * g.d * 2;
    int e = make_tmap_bf16_3d(&tk, K_ev, g.d, (uint64_t)n_ev, g.BH, (uint64_t)g.d * 2, hs, 64, AbsCfg<128>::TT);
    if (e) return e;
    e = make_tmap_bf16_3d(&tv, V_ev, g.d, (uint64_t)n_ev, g.BH, (uint64_t)g.d * 2, hs, 64, AbsCfg<128>::TT);
    if (e) return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int n_tiles = (n_ev + AbsCfg<128>::TT - 1) / AbsCfg<128>::TT;
    int CL = sms / (g.BH > 0 ? g.BH : 1);
    CL = CL < 1 ? 1 : (CL > 8 ? 8 : CL);
    CL = CL > n_tiles ? n_tiles : CL;
    AbsParams p{g.BH, n_ev, CL, S, z, status, wait_limit_ns};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return g.d == 128 ? launch_absorb_t<128>(tk, tv, p, st) : launch_absorb_t<64>(tk, tv, p, st);
}

}  // namespace hf
