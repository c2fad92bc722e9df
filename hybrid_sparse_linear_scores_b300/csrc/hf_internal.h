// hf_internal.h -- definitions shared by the library's .cu files (never by
// the oracle): device error codes, derived geometry, kernel parameter blocks,
// workspace layout and the launch functions each .cu file provides.
#pragma once

#include <cstddef>
#include <cstdint>

#include "hf.h"

namespace hf {

// Device status word codes (match hf_status values).
constexpr uint32_t HF_DEV_ERR_TIMEOUT = 4;
constexpr uint32_t HF_DEV_ERR_CHECK = 5;

// Wait / check sites reported with a device error.
enum Site : uint32_t {
    SITE_ATTN_Q = 101,
    SITE_ATTN_KV_FULL = 102,
    SITE_ATTN_KV_EMPTY = 103,
    SITE_ATTN_S_FULL = 104,
    SITE_ATTN_P_FULL = 105,
    SITE_ATTN_PV_DONE = 106,
    SITE_ATTN_LIN = 107,
    SITE_ATTN_PHIQ = 108,
    SITE_ATTN_DRAIN = 109,
    SITE_ATTN_BAD_INDEX = 110,
    SITE_ABSORB_FULL = 201,
    SITE_ABSORB_EMPTY = 202,
    SITE_ABSORB_PHI = 203,
    SITE_ABSORB_ACC = 204,
    SITE_ABSORB_DRAIN = 205,
    SITE_SELFTEST = 301,
    SITE_PROLOGUE_Q = 401,
    SITE_POOL_KEYS = 402,
};

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;   // 2 s

struct SlotMap {
    int32_t s[HF_MAX_WINDOW_FRAMES];
};

// What a pooling launch covers: the chunk's query blocks (with_q) and the
// key blocks of the ring slots slot[0..n).
struct PoolFrames {
    int32_t slot[HF_MAX_WINDOW_FRAMES];
    int32_t n;
    int32_t with_q;
};

// Geometry of one call, derived and validated on the host.
struct Geom {
    int32_t BH;          // batch * heads
    int32_t d;           // head_dim
    int32_t nf;          // tokens per frame
    int32_t C;           // chunk frames
    int32_t W;           // ring slots
    int32_t n_win;       // frames in the window now
    int32_t beta;        // block size
    int32_t bpf;         // blocks per frame
    int32_t nqb;         // query blocks (C * bpf)
    int32_t nkb;         // key blocks (n_win * bpf)
    int32_t k_eff;       // min(topk, nkb)
    int32_t slot_stride; // rows per ring slot
    float scale_log2;    // softmax scale * log2(e)
    float eps;           // linear-read epsilon
};

// Workspace layout (byte offsets, 1024-aligned).
struct WsLayout {
    size_t status;   // 256 B: uint32 [0] code, [1] site
    size_t counters; // uint32 [BH * pairs per head][2]: parts of a split pair that arrived (zero between calls)
    size_t qp;       // fp32 [BH][nQB][d] (hf_block_scores)
    size_t kp;       // fp32 [BH][W slots][d/4][bpf][4]: pooled keys of every ring slot (kept between calls)
    size_t smma;     // bf16 [BH][2][d*d]  (S hi / lo, MMA operand layout; kept between calls)
    size_t idx;      // int32 [BH][nQB][K_max] (the only region whose size follows topk)
    size_t prounds;  // int32 [BH * pairs per head]: weight of each tile pair's slab stream
    size_t total_compact;   // end of the above: the attention runs without splitting pairs
    size_t partial;  // fp32 [kAttnMaxGrid][2][2][128][d + 4]: partial results of split pairs
    size_t total;
};

// Balancing weight of one round of a tile pair's slab stream, in the units of
// the attention kernel's equal shares per CTA: a fixed part plus the MMAs of
// each tile that takes part in the round (4 per slab of P V, 8 of Q K^T),
// halved.  sa, sb: slabs of the round that tile A / tile B needs (0..2).  A
// round of both tiles costs about 1.35 times a round of one tile.
__host__ __device__ constexpr uint32_t round_weight(int sa, int sb)
{
    return 15u + (sa ? 2u * (uint32_t)sa + 4u : 0u) + (sb ? 2u * (uint32_t)sb + 4u : 0u);
}
// Units charged to each pair part on top of its rounds (epilogue and slab
// list: about six rounds of both tiles; 160-200 measured best, 248 and 300
// slower by 1 and 4 us on the realistic layer).
constexpr uint32_t kPartWeight = 192;

// Largest attention grid (one CTA per SM, at most this many): the partial
// results of split pairs are sized for it.
constexpr int kAttnMaxGrid = 160;

// ---- launchers (return cudaError_t as int) --------------------------------
int launch_pool(const uint16_t* Q, const uint16_t* Kc, const Geom& g, const PoolFrames& pf, float* qp, float* kpc,
                void* stream);
// Scores of pooled query blocks qp [BH][nQB][d] against the window's cached
// key pools (the standalone hf_block_scores).
int launch_scores(const float* qp, const float* kpc, const Geom& g, const SlotMap& sm, float* scores, void* stream);
int launch_topk(const float* scores, const Geom& g, int32_t* idx, void* stream);
// The hybrid forward's prologue in one launch: pooling of the chunk's query
// blocks, the state as the epilogue's tensor-core operand (S -> bf16 hi/lo),
// scores against the cached key pools, top-K and, when pair_rounds is given,
// each tile pair's weight (and its arrival counters zeroed).  after_pool: the
// kernel launched just before on `stream` is a key pooling, and the prologue
// may start while it runs (it reads Q and S meanwhile, the pooled keys only
// after waiting for it).
int launch_fwd_prologue(const uint16_t* Q, const float* kpc, const float* S, const Geom& g, const SlotMap& sm,
                        int32_t* idx, uint16_t* smma, int32_t* pair_rounds, uint32_t* counters, uint32_t* status,
                        uint64_t wait_limit_ns, bool after_pool, void* stream);
// Key-block pooling of ring slots pf.slot[0..pf.n) into the cache, bulk copies.
int launch_pool_keys(const uint16_t* Kc, const Geom& g, const PoolFrames& pf, float* kpc, uint32_t* status,
                     uint64_t wait_limit_ns, void* stream);
int launch_attn(const uint16_t* Q, const uint16_t* Kc, const uint16_t* Vc, const Geom& g, const SlotMap& sm,
                const int32_t* idx, const uint16_t* smma, const float* z, float* o_swa, uint16_t* o_bf16,
                const int32_t* pair_rounds, float* partial, uint32_t* counters, uint32_t* status,
                uint64_t wait_limit_ns, void* stream);

// Relative temporal RoPE pre-step: element (h, f, t, c) at
// h * head_stride + slot[f] * frame_stride + t * d + c (src and dst alike).
struct RopeParams {
    const uint16_t* src;
    uint16_t* dst;
    int64_t head_stride, frame_stride;      // elements
    int BH, n_frames, nf, d, rot_dims;
    int32_t slot[HF_MAX_WINDOW_FRAMES];     // frame f's position along frame_stride
    int32_t pos[HF_MAX_WINDOW_FRAMES];      // frame f's clamped offset
    float inv_freq[64];                     // base^(-2i / rot_dims), i < rot_dims / 2
};
int launch_rope(const RopeParams& p, void* stream);
int launch_linear_read(const uint16_t* Q, const float* S, const float* z, const Geom& g, float* O, int accumulate,
                       void* stream);
int launch_absorb(const uint16_t* K_ev, const uint16_t* V_ev, int32_t n_ev, int64_t head_stride, const Geom& g,
                  float* S, float* z, uint16_t* smma, bool share_sms, uint32_t* status, uint64_t wait_limit_ns,
                  void* stream);
int launch_state_reset(float* S, float* z, const Geom& g, void* stream);
int launch_selftest_wait(uint32_t* status, uint64_t limit_ns, void* stream);

// The hybrid forward behind hf_hybrid_forward_ex.  allow_split = false runs
// the attention without cutting tile pairs between CTAs, for a workspace of
// compact_workspace_bytes() (no partial-result buffer).
hf_status forward_impl(const hf_config* cfg, const uint16_t* Q, const uint16_t* Kc, const uint16_t* Vc,
                       int32_t slot_stride, const int32_t* slot_map, int32_t n_win, const float* S, const float* z,
                       uint16_t* O, int32_t* idx_out, void* ws, void* stream, uint32_t flags, void* const* events,
                       void* state_ready, bool allow_split);
size_t compact_workspace_bytes(const hf_config* cfg);

// Records a printf-style message as the calling thread's hf_last_error()
// text and returns `code`.
hf_status set_last_error(hf_status code, const char* fmt, ...);

// Host helper: cuTensorMapEncodeTiled for a 3-D bf16 tensor with a
// 128-byte swizzle.  dims/strides in elements/bytes (innermost first).
int make_tmap_bf16_3d(void* tmap_out, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                      uint64_t stride2_bytes, uint32_t box0, uint32_t box1);

}  // namespace hf
