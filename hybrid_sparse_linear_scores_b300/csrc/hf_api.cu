// hf_api.cu -- the C ABI declared in include/hf.h: argument validation,
// workspace layout, tensor-map encoding and the launch sequence of each
// entry point.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "hf.h"
#include "hf_internal.h"

namespace hf {
namespace {

thread_local char g_last_error[256] = "";

hf_status fail(hf_status s, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

hf_status cuda_fail(int err, const char* what)
{
    return fail(HF_ERR_CUDA, "%s: %s", what, cudaGetErrorString(static_cast<cudaError_t>(err)));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align1k(size_t x) { return (x + 1023) & ~size_t(1023); }

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ---- config ---------------------------------------------------------------
hf_status check_cfg(const hf_config* cfg)
{
    if (!cfg) return fail(HF_ERR_INVALID_ARG, "cfg is NULL");
    if (cfg->batch < 1 || cfg->heads < 1) return fail(HF_ERR_INVALID_ARG, "batch and heads must be >= 1");
    if (cfg->head_dim != 64 && cfg->head_dim != 128)
        return fail(HF_ERR_UNSUPPORTED, "head_dim %d not in {64, 128}", cfg->head_dim);
    if (cfg->tokens_per_frame < 1) return fail(HF_ERR_INVALID_ARG, "tokens_per_frame must be >= 1");
    if (cfg->window_frames < 1 || cfg->window_frames > HF_MAX_WINDOW_FRAMES)
        return fail(HF_ERR_UNSUPPORTED, "window_frames %d not in [1, %d]", cfg->window_frames, HF_MAX_WINDOW_FRAMES);
    if (cfg->chunk_frames < 1 || cfg->chunk_frames > cfg->window_frames)
        return fail(HF_ERR_INVALID_ARG, "chunk_frames %d not in [1, window_frames]", cfg->chunk_frames);
    if (cfg->block_size != 32 && cfg->block_size != 64 && cfg->block_size != 128)
        return fail(HF_ERR_UNSUPPORTED, "block_size %d not in {32, 64, 128}", cfg->block_size);
    if (cfg->topk < 1) return fail(HF_ERR_INVALID_ARG, "topk must be >= 1");
    if (!(cfg->softmax_scale >= 0.0f) || !std::isfinite(cfg->softmax_scale))
        return fail(HF_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
    if (!(cfg->lin_eps >= 0.0f) || !std::isfinite(cfg->lin_eps))
        return fail(HF_ERR_INVALID_ARG, "lin_eps must be finite and >= 0");
    const long bpf = ceil_div(cfg->tokens_per_frame, cfg->block_size);
    if (bpf * cfg->window_frames > HF_MAX_KEY_BLOCKS)
        return fail(HF_ERR_UNSUPPORTED, "window has %ld key blocks (> %d)", bpf * cfg->window_frames,
                    HF_MAX_KEY_BLOCKS);
    if ((long)cfg->batch * cfg->heads > (1L << 20)) return fail(HF_ERR_UNSUPPORTED, "batch*heads too large");
    return HF_OK;
}

Geom make_geom(const hf_config* cfg, int n_win, int slot_stride)
{
    Geom g;
    g.BH = cfg->batch * cfg->heads;
    g.d = cfg->head_dim;
    g.nf = cfg->tokens_per_frame;
    g.C = cfg->chunk_frames;
    g.W = cfg->window_frames;
    g.n_win = n_win;
    g.beta = cfg->block_size;
    g.bpf = ceil_div(g.nf, g.beta);
    g.nqb = g.C * g.bpf;
    g.nkb = n_win * g.bpf;
    g.k_eff = cfg->topk < g.nkb ? cfg->topk : g.nkb;
    g.slot_stride = slot_stride;
    const float scale = cfg->softmax_scale > 0.0f ? cfg->softmax_scale : 1.0f / std::sqrt((float)g.d);
    g.scale_log2 = scale * 1.4426950408889634f;
    g.eps = cfg->lin_eps;
    return g;
}

WsLayout ws_layout(const hf_config* cfg)
{
    const size_t BH = (size_t)cfg->batch * cfg->heads;
    const size_t d = (size_t)cfg->head_dim;
    const size_t bpf = (size_t)ceil_div(cfg->tokens_per_frame, cfg->block_size);
    const size_t nqb = (size_t)cfg->chunk_frames * bpf;
    const size_t nkb = (size_t)cfg->window_frames * bpf;
    const size_t kmax = (size_t)cfg->topk < nkb ? (size_t)cfg->topk : nkb;
    const size_t G = (size_t)(128 / cfg->block_size);             // query blocks per tile
    const size_t pairs = BH * ((ceil_div((int)nqb, (int)G) + 1) / 2);
    WsLayout w;
    // the status word and the split counters (both zero between calls) come
    // first, where a change of topk between calls does not move them
    w.status = 0;
    w.counters = 1024;
    w.qp = w.counters + align1k(pairs * 2 * 4);
    w.kp = w.qp + align1k(BH * nqb * d * 4);
    // the pooled-key cache and the state operand persist between calls, so they
    // come before the one region whose size follows topk
    w.smma = w.kp + align1k(BH * nkb * d * 4);
    w.idx = w.smma + align1k(BH * 2 * d * d * 2);
    w.prounds = w.idx + align1k(BH * nqb * kmax * 4);
    w.total_compact = w.prounds + align1k(pairs * 4);
    w.partial = w.total_compact;
    w.total = w.partial + (size_t)HF_SPLIT_PARTIAL_BYTES(d);
    static_assert(HF_SPLIT_PARTIAL_BYTES(0) == (size_t)kAttnMaxGrid * 2 * 2 * 128 * 4 * 4, "split buffer sizing");
    return w;
}

// ---- window arguments -------------------------------------------------------
hf_status check_window(const hf_config* cfg, int32_t slot_stride, const int32_t* slot_map, int32_t n_win,
                       SlotMap* sm)
{
    if (n_win < cfg->chunk_frames || n_win > cfg->window_frames)
        return fail(HF_ERR_INVALID_ARG, "n_win %d not in [chunk_frames %d, window_frames %d]", n_win,
                    cfg->chunk_frames, cfg->window_frames);
    if (slot_stride < cfg->tokens_per_frame)
        return fail(HF_ERR_INVALID_ARG, "slot_stride %d < tokens_per_frame %d", slot_stride, cfg->tokens_per_frame);
    uint64_t used = 0;
    for (int w = 0; w < HF_MAX_WINDOW_FRAMES; ++w) sm->s[w] = 0;
    for (int w = 0; w < n_win; ++w) {
        const int s = slot_map ? slot_map[w] : w;
        if (s < 0 || s >= cfg->window_frames)
            return fail(HF_ERR_INVALID_ARG, "slot_map[%d] = %d outside [0, %d)", w, s, cfg->window_frames);
        if (used & (1ull << s)) return fail(HF_ERR_INVALID_ARG, "slot_map[%d] = %d used twice", w, s);
        used |= 1ull << s;
        sm->s[w] = s;
    }
    return HF_OK;
}

// Pool the chunk's queries and the keys of every frame of the window.
PoolFrames window_frames(const SlotMap& sm, int n_win)
{
    PoolFrames pf;
    for (int w = 0; w < HF_MAX_WINDOW_FRAMES; ++w) pf.slot[w] = w < n_win ? sm.s[w] : 0;
    pf.n = n_win;
    pf.with_q = 1;
    return pf;
}

#define HF_CHECK_PTR(p)                                                                          \
    do {                                                                                         \
        if (!(p)) return fail(HF_ERR_INVALID_ARG, "%s is NULL", #p);                             \
        if (!aligned16(p)) return fail(HF_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p);     \
    } while (0)

#define HF_LAUNCH(expr, what)                                 \
    do {                                                      \
        const int e_ = (expr);                                \
        if (e_ != 0) return cuda_fail(e_, what);              \
    } while (0)

// ---- tensor maps ------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

hf_status set_last_error(hf_status code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

int make_tmap_bf16_3d(void* tmap_out, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                      uint64_t stride2_bytes, uint32_t box0, uint32_t box1)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return (int)cudaErrorNotSupported;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {box0, box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(static_cast<CUtensorMap*>(tmap_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

}  // namespace hf

using namespace hf;

extern "C" {

int32_t hf_abi_version(void) { return HF_ABI_VERSION; }

const char* hf_status_string(hf_status s)
{
    switch (s) {
    case HF_OK: return "HF_OK";
    case HF_ERR_INVALID_ARG: return "HF_ERR_INVALID_ARG";
    case HF_ERR_UNSUPPORTED: return "HF_ERR_UNSUPPORTED";
    case HF_ERR_CUDA: return "HF_ERR_CUDA";
    case HF_ERR_TIMEOUT: return "HF_ERR_TIMEOUT";
    case HF_ERR_DEVICE_CHECK: return "HF_ERR_DEVICE_CHECK";
    }
    return "unknown hf_status";
}

const char* hf_last_error(void) { return g_last_error; }

hf_status hf_workspace_size(const hf_config* cfg, size_t* bytes)
{
    hf_status s = check_cfg(cfg);
    if (s != HF_OK) return s;
    if (!bytes) return fail(HF_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = ws_layout(cfg).total;
    return HF_OK;
}

hf_status hf_state_reset(const hf_config* cfg, float* S, float* z, void* stream)
{
    hf_status s = check_cfg(cfg);
    if (s != HF_OK) return s;
    HF_CHECK_PTR(S);
    HF_CHECK_PTR(z);
    const Geom g = make_geom(cfg, cfg->chunk_frames, cfg->tokens_per_frame);
    HF_LAUNCH(launch_state_reset(S, z, g, stream), "state reset launch");
    return HF_OK;
}

hf_status hf_absorb_evicted_strided(const hf_config* cfg, float* S, float* z, const uint16_t* K_ev,
                                    const uint16_t* V_ev, int32_t n_ev_tokens, int64_t head_stride_tokens, void* ws,
                                    void* stream, uint32_t flags)
{
    hf_status s = check_cfg(cfg);
    if (s != HF_OK) return s;
    if (flags & ~(uint32_t)HF_ABSORB_SHARE_SMS) return fail(HF_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    if (n_ev_tokens < 0) return fail(HF_ERR_INVALID_ARG, "n_ev_tokens %d < 0", n_ev_tokens);
    if (head_stride_tokens < n_ev_tokens)
        return fail(HF_ERR_INVALID_ARG, "head_stride_tokens %lld < n_ev_tokens %d", (long long)head_stride_tokens,
                    n_ev_tokens);
    HF_CHECK_PTR(S);
    HF_CHECK_PTR(z);
    HF_CHECK_PTR(ws);
    if (n_ev_tokens == 0) return HF_OK;
    HF_CHECK_PTR(K_ev);
    HF_CHECK_PTR(V_ev);
    const Geom g = make_geom(cfg, cfg->chunk_frames, cfg->tokens_per_frame);
    const WsLayout L = ws_layout(cfg);
    uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + L.status);
    // the new S also goes to the workspace as the linear read's MMA operand, so
    // that a forward with HF_FWD_STATE_PREPARED need not read S
    uint16_t* smma = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + L.smma);
    HF_LAUNCH(launch_absorb(K_ev, V_ev, n_ev_tokens, head_stride_tokens, g, S, z, smma,
                            (flags & HF_ABSORB_SHARE_SMS) != 0, status, kDefaultWaitLimitNs, stream),
              "absorb launch");
    return HF_OK;
}

hf_status hf_absorb_evicted(const hf_config* cfg, float* S, float* z, const uint16_t* K_ev, const uint16_t* V_ev,
                            int32_t n_ev_tokens, void* ws, void* stream)
{
    return hf_absorb_evicted_strided(cfg, S, z, K_ev, V_ev, n_ev_tokens, n_ev_tokens, ws, stream, 0u);
}

hf_status hf_block_scores(const hf_config* cfg, const uint16_t* Q, const uint16_t* Kc, int32_t slot_stride,
                          const int32_t* slot_map, int32_t n_win, float* scores, void* ws, void* stream)
{
    hf_status s = check_cfg(cfg);
    if (s != HF_OK) return s;
    HF_CHECK_PTR(Q);
    HF_CHECK_PTR(Kc);
    HF_CHECK_PTR(scores);
    HF_CHECK_PTR(ws);
    SlotMap sm;
    if ((s = check_window(cfg, slot_stride, slot_map, n_win, &sm)) != HF_OK) return s;
    const Geom g = make_geom(cfg, n_win, slot_stride);
    const WsLayout L = ws_layout(cfg);
    uint8_t* w = static_cast<uint8_t*>(ws);
    float* qp = reinterpret_cast<float*>(w + L.qp);
    float* kp = reinterpret_cast<float*>(w + L.kp);
    HF_LAUNCH(launch_pool(Q, Kc, g, window_frames(sm, n_win), qp, kp, stream), "pool launch");
    HF_LAUNCH(launch_scores(qp, kp, g, sm, scores, stream), "score launch");
    return HF_OK;
}

hf_status hf_topk_blocks(const hf_config* cfg, const float* scores, int32_t nQB, int32_t nKB, int32_t* idx,
                         void* stream)
{
    hf_status s = check_cfg(cfg);
    if (s != HF_OK) return s;
    HF_CHECK_PTR(scores);
    HF_CHECK_PTR(idx);
    if (nQB < 1 || nKB < 1) return fail(HF_ERR_INVALID_ARG, "nQB and nKB must be >= 1");
    if (nKB > HF_MAX_KEY_BLOCKS) return fail(HF_ERR_UNSUPPORTED, "nKB %d > %d", nKB, HF_MAX_KEY_BLOCKS);
    Geom g = make_geom(cfg, cfg->chunk_frames, cfg->tokens_per_frame);
    g.nqb = nQB;
    g.nkb = nKB;
    g.k_eff = cfg->topk < nKB ? cfg->topk : nKB;
    HF_LAUNCH(launch_topk(scores, g, idx, stream), "top-k launch");
    return HF_OK;
}

hf_status hf_sparse_swa_attn(const hf_config* cfg, const uint16_t* Q, const uint16_t* Kc, const uint16_t* Vc,
                             int32_t slot_stride, const int32_t* slot_map, int32_t n_win, const int32_t* idx,
                             float* O_swa, void* ws, void* stream)
{
    hf_status s = check_cfg(cfg);
    if (s != HF_OK) return s;
    HF_CHECK_PTR(Q);
    HF_CHECK_PTR(Kc);
    HF_CHECK_PTR(Vc);
    HF_CHECK_PTR(idx);
    HF_CHECK_PTR(O_swa);
    HF_CHECK_PTR(ws);
    SlotMap sm;
    if ((s = check_window(cfg, slot_stride, slot_map, n_win, &sm)) != HF_OK) return s;
    const Geom g = make_geom(cfg, n_win, slot_stride);
    uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + ws_layout(cfg).status);
    HF_LAUNCH(launch_attn(Q, Kc, Vc, g, sm, idx, nullptr, nullptr, O_swa, nullptr, nullptr, nullptr, nullptr, status,
                          kDefaultWaitLimitNs, stream),
              "sparse attention launch");
    return HF_OK;
}

hf_status hf_linear_read(const hf_config* cfg, const uint16_t* Q, const float* S, const float* z, float* O,
                         int32_t accumulate, void* stream)
{
    hf_status s = check_cfg(cfg);
    if (s != HF_OK) return s;
    HF_CHECK_PTR(Q);
    HF_CHECK_PTR(S);
    HF_CHECK_PTR(z);
    HF_CHECK_PTR(O);
    const Geom g = make_geom(cfg, cfg->chunk_frames, cfg->tokens_per_frame);
    HF_LAUNCH(launch_linear_read(Q, S, z, g, O, accumulate, stream), "linear read launch");
    return HF_OK;
}

}  // extern "C"

namespace hf {

size_t compact_workspace_bytes(const hf_config* cfg) { return ws_layout(cfg).total_compact; }

hf_status forward_impl(const hf_config* cfg, const uint16_t* Q, const uint16_t* Kc, const uint16_t* Vc,
                       int32_t slot_stride, const int32_t* slot_map, int32_t n_win, const float* S, const float* z,
                       uint16_t* O, int32_t* idx_out, void* ws, void* stream, uint32_t flags, void* const* events,
                       void* state_ready, bool allow_split)
{
    hf_status s = check_cfg(cfg);
    if (s != HF_OK) return s;
    if (flags & ~(uint32_t)(HF_FWD_CACHED_KEYS | HF_FWD_STATE_PREPARED | HF_FWD_AFTER_POOL_KEYS))
        return fail(HF_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    const bool prepared = (flags & HF_FWD_STATE_PREPARED) != 0;
    HF_CHECK_PTR(Q);
    HF_CHECK_PTR(Kc);
    HF_CHECK_PTR(Vc);
    if (!prepared) HF_CHECK_PTR(S);
    HF_CHECK_PTR(z);
    HF_CHECK_PTR(O);
    HF_CHECK_PTR(ws);
    if (idx_out && !aligned16(idx_out)) return fail(HF_ERR_INVALID_ARG, "idx_out is not 16-byte aligned");
    SlotMap sm;
    if ((s = check_window(cfg, slot_stride, slot_map, n_win, &sm)) != HF_OK) return s;
    const Geom g = make_geom(cfg, n_win, slot_stride);
    const WsLayout L = ws_layout(cfg);
    uint8_t* w = static_cast<uint8_t*>(ws);
    float* kp = reinterpret_cast<float*>(w + L.kp);
    int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(w + L.idx);
    uint16_t* smma = reinterpret_cast<uint16_t*>(w + L.smma);
    uint32_t* status = reinterpret_cast<uint32_t*>(w + L.status);
    // Cutting tile pairs between CTAs balances weighted rounds in 32-bit unit
    // counts: at most round_weight(2, 2) per round and kPartWeight per pair.
    // Layers too large for that (far beyond a realistic layer) run whole pairs.
    {
        const long per_tile = 128 / g.beta;
        const long pairs = (long)g.BH * ((((long)g.nqb + per_tile - 1) / per_tile + 1) / 2);
        const long max_rounds = ((long)g.n_win * ((g.nf + 63) / 64) + 1) / 2;
        if (pairs * ((long)round_weight(2, 2) * max_rounds + (long)kPartWeight) >= (1L << 31)) allow_split = false;
    }
    int32_t* prounds = allow_split ? reinterpret_cast<int32_t*>(w + L.prounds) : nullptr;
    float* partial = allow_split ? reinterpret_cast<float*>(w + L.partial) : nullptr;
    uint32_t* counters = allow_split ? reinterpret_cast<uint32_t*>(w + L.counters) : nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // inside a stream capture an event becomes an external record node, so that it
    // also times the graph's replays
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    if (events && cudaStreamIsCapturing(st, &capturing) != cudaSuccess) capturing = cudaStreamCaptureStatusNone;
    auto mark = [&](int i) -> int {
        if (!events || !events[i]) return 0;
        cudaEvent_t e = static_cast<cudaEvent_t>(events[i]);
        return capturing == cudaStreamCaptureStatusActive
                   ? (int)cudaEventRecordWithFlags(e, st, cudaEventRecordExternal)
                   : (int)cudaEventRecord(e, st);
    };
    PoolFrames pf = window_frames(sm, n_win);
    pf.with_q = 0;
    if (flags & HF_FWD_CACHED_KEYS) pf.n = 0;   // the window's key blocks are already in the cache
    HF_LAUNCH(mark(0), "event record");
    HF_LAUNCH(launch_pool_keys(Kc, g, pf, kp, status, kDefaultWaitLimitNs, stream), "key pooling launch");
    HF_LAUNCH(mark(1), "event record");
    // the prologue converts S into the state operand unless the workspace already
    // holds it (HF_FWD_STATE_PREPARED: written by the absorb that produced S)
    // the prologue may start while a key pooling launched just before it runs:
    // the one above, or (HF_FWD_AFTER_POOL_KEYS) the caller's hf_pool_keys
    const bool after_pool = pf.n > 0 || (flags & HF_FWD_AFTER_POOL_KEYS) != 0;
    HF_LAUNCH(launch_fwd_prologue(Q, kp, prepared ? nullptr : S, g, sm, idx, smma, prounds, counters, status,
                                  kDefaultWaitLimitNs, after_pool, stream),
              "prologue launch");
    HF_LAUNCH(mark(2), "event record");
    // only the attention kernel reads the state (operand and z): it may wait for
    // the absorb that the prologue did not need to wait for
    if (state_ready)
        HF_LAUNCH((int)cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(state_ready), 0), "state-ready event wait");
    HF_LAUNCH(launch_attn(Q, Kc, Vc, g, sm, idx, smma, z, nullptr, O, prounds, partial, counters, status,
                          kDefaultWaitLimitNs, stream),
              "hybrid attention launch");
    HF_LAUNCH(mark(3), "event record");
    return HF_OK;
}

}  // namespace hf

extern "C" {

hf_status hf_hybrid_forward_ex(const hf_config* cfg, const uint16_t* Q, const uint16_t* Kc, const uint16_t* Vc,
                               int32_t slot_stride, const int32_t* slot_map, int32_t n_win, const float* S,
                               const float* z, uint16_t* O, int32_t* idx_out, void* ws, void* stream, uint32_t flags,
                               void* const* events, void* state_ready)
{
    return forward_impl(cfg, Q, Kc, Vc, slot_stride, slot_map, n_win, S, z, O, idx_out, ws, stream, flags, events,
                        state_ready, true);
}

hf_status hf_hybrid_forward_profiled(const hf_config* cfg, const uint16_t* Q, const uint16_t* Kc, const uint16_t* Vc,
                                     int32_t slot_stride, const int32_t* slot_map, int32_t n_win, const float* S,
                                     const float* z, uint16_t* O, int32_t* idx_out, void* ws, void* stream,
                                     void* const* events)
{
    return hf_hybrid_forward_ex(cfg, Q, Kc, Vc, slot_stride, slot_map, n_win, S, z, O, idx_out, ws, stream, 0u,
                                events, nullptr);
}

hf_status hf_hybrid_forward(const hf_config* cfg, const uint16_t* Q, const uint16_t* Kc, const uint16_t* Vc,
                            int32_t slot_stride, const int32_t* slot_map, int32_t n_win, const float* S,
                            const float* z, uint16_t* O, int32_t* idx_out, void* ws, void* stream)
{
    return hf_hybrid_forward_ex(cfg, Q, Kc, Vc, slot_stride, slot_map, n_win, S, z, O, idx_out, ws, stream, 0u,
                                nullptr, nullptr);
}

hf_status hf_rope_relative(const hf_config* cfg, const uint16_t* src, uint16_t* dst, int64_t head_stride,
                           int64_t frame_stride, const int32_t* slots, const int32_t* offsets, int32_t n_frames,
                           int32_t max_offset, int32_t rot_dims, float theta_base, void* stream)
{
    hf_status s = check_cfg(cfg);
    if (s != HF_OK) return s;
    HF_CHECK_PTR(src);
    HF_CHECK_PTR(dst);
    const int d = cfg->head_dim;
    if (n_frames < 1 || n_frames > HF_MAX_WINDOW_FRAMES)
        return fail(HF_ERR_INVALID_ARG, "n_frames %d not in [1, %d]", n_frames, HF_MAX_WINDOW_FRAMES);
    if (!slots || !offsets) return fail(HF_ERR_INVALID_ARG, "slots / offsets is NULL");
    if (rot_dims < 0 || rot_dims > d || rot_dims % 8 != 0)
        return fail(HF_ERR_INVALID_ARG, "rot_dims %d not a multiple of 8 in [0, head_dim %d]", rot_dims, d);
    if (max_offset < 0) return fail(HF_ERR_INVALID_ARG, "max_offset %d < 0", max_offset);
    if (!(theta_base > 1.0f) || !(theta_base < 3.0e38f))
        return fail(HF_ERR_INVALID_ARG, "theta_base must be finite and > 1");
    if (head_stride % 8 != 0 || frame_stride % 8 != 0)
        return fail(HF_ERR_INVALID_ARG, "strides must be multiples of 8 elements");
    if (frame_stride < (int64_t)cfg->tokens_per_frame * d)
        return fail(HF_ERR_INVALID_ARG, "frame_stride %lld < tokens_per_frame * head_dim",
                    (long long)frame_stride);
    RopeParams p;
    p.src = src;
    p.dst = dst;
    p.head_stride = head_stride;
    p.frame_stride = frame_stride;
    p.BH = cfg->batch * cfg->heads;
    p.n_frames = n_frames;
    p.nf = cfg->tokens_per_frame;
    p.d = d;
    p.rot_dims = rot_dims;
    uint64_t used = 0;
    int32_t max_slot = 0;
    for (int f = 0; f < n_frames; ++f) {
        if (slots[f] < 0 || slots[f] >= 64) return fail(HF_ERR_INVALID_ARG, "slots[%d] = %d outside [0, 64)", f, slots[f]);
        if (used & (1ull << slots[f])) return fail(HF_ERR_INVALID_ARG, "slots[%d] = %d given twice", f, slots[f]);
        used |= 1ull << slots[f];
        max_slot = slots[f] > max_slot ? slots[f] : max_slot;
        p.slot[f] = slots[f];
        p.pos[f] = offsets[f] < 0 ? 0 : (offsets[f] > max_offset ? max_offset : offsets[f]);
    }
    if (head_stride < (int64_t)(max_slot + 1) * frame_stride)
        return fail(HF_ERR_INVALID_ARG, "head_stride %lld smaller than the frames it holds", (long long)head_stride);
    for (int i = 0; i < 64; ++i)
        p.inv_freq[i] = i < rot_dims / 2 ? (float)pow((double)theta_base, -2.0 * i / rot_dims) : 0.0f;
    HF_LAUNCH(launch_rope(p, stream), "rope launch");
    return HF_OK;
}

hf_status hf_ring_write(const hf_config* cfg, const uint16_t* K_src, const uint16_t* V_src, uint16_t* Kc, uint16_t* Vc,
                        int32_t slot_stride, const int32_t* slots, int32_t n_frames, void* stream)
{
    hf_status s = check_cfg(cfg);
    if (s != HF_OK) return s;
    HF_CHECK_PTR(K_src);
    HF_CHECK_PTR(V_src);
    HF_CHECK_PTR(Kc);
    HF_CHECK_PTR(Vc);
    if (n_frames < 1 || n_frames > cfg->window_frames)
        return fail(HF_ERR_INVALID_ARG, "n_frames %d not in [1, window_frames %d]", n_frames, cfg->window_frames);
    if (slot_stride < cfg->tokens_per_frame)
        return fail(HF_ERR_INVALID_ARG, "slot_stride %d < tokens_per_frame %d", slot_stride, cfg->tokens_per_frame);
    if (!slots) return fail(HF_ERR_INVALID_ARG, "slots is NULL");
    uint64_t used = 0;
    for (int i = 0; i < n_frames; ++i) {
        const int sl = slots[i];
        if (sl < 0 || sl >= cfg->window_frames)
            return fail(HF_ERR_INVALID_ARG, "slots[%d] = %d outside [0, %d)", i, sl, cfg->window_frames);
        if (used & (1ull << sl)) return fail(HF_ERR_INVALID_ARG, "slots[%d] = %d given twice", i, sl);
        used |= 1ull << sl;
    }
    const size_t BH = (size_t)cfg->batch * cfg->heads;
    const size_t d = (size_t)cfg->head_dim;
    const size_t frame = (size_t)cfg->tokens_per_frame * d;                 // elements of one frame of one head
    const size_t spitch = (size_t)n_frames * frame * 2;                     // bytes between heads in the source
    const size_t dpitch = (size_t)cfg->window_frames * slot_stride * d * 2; // bytes between heads in the ring
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int f = 0; f < n_frames; ++f) {
        const size_t doff = (size_t)slots[f] * slot_stride * d;
        HF_LAUNCH(cudaMemcpy2DAsync(Kc + doff, dpitch, K_src + f * frame, spitch, frame * 2, BH, cudaMemcpyDefault, st),
                  "ring write (K)");
        HF_LAUNCH(cudaMemcpy2DAsync(Vc + doff, dpitch, V_src + f * frame, spitch, frame * 2, BH, cudaMemcpyDefault, st),
                  "ring write (V)");
    }
    return HF_OK;
}

hf_status hf_pool_keys(const hf_config* cfg, const uint16_t* Kc, int32_t slot_stride, const int32_t* slots,
                       int32_t n_slots, void* ws, void* stream)
{
    hf_status s = check_cfg(cfg);
    if (s != HF_OK) return s;
    HF_CHECK_PTR(Kc);
    HF_CHECK_PTR(ws);
    if (n_slots < 0 || n_slots > cfg->window_frames)
        return fail(HF_ERR_INVALID_ARG, "n_slots %d not in [0, window_frames %d]", n_slots, cfg->window_frames);
    if (slot_stride < cfg->tokens_per_frame)
        return fail(HF_ERR_INVALID_ARG, "slot_stride %d < tokens_per_frame %d", slot_stride, cfg->tokens_per_frame);
    if (n_slots > 0 && !slots) return fail(HF_ERR_INVALID_ARG, "slots is NULL");
    PoolFrames pf;
    uint64_t used = 0;
    for (int i = 0; i < HF_MAX_WINDOW_FRAMES; ++i) pf.slot[i] = 0;
    for (int i = 0; i < n_slots; ++i) {
        const int sl = slots[i];
        if (sl < 0 || sl >= cfg->window_frames)
            return fail(HF_ERR_INVALID_ARG, "slots[%d] = %d outside [0, %d)", i, sl, cfg->window_frames);
        if (used & (1ull << sl)) return fail(HF_ERR_INVALID_ARG, "slots[%d] = %d given twice", i, sl);
        used |= 1ull << sl;
        pf.slot[i] = sl;
    }
    pf.n = n_slots;
    pf.with_q = 0;
    if (n_slots == 0) return HF_OK;
    const Geom g = make_geom(cfg, cfg->chunk_frames, slot_stride);
    const WsLayout L = ws_layout(cfg);
    float* kp = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + L.kp);
    uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + L.status);
    HF_LAUNCH(launch_pool_keys(Kc, g, pf, kp, status, kDefaultWaitLimitNs, stream), "key pool launch");
    return HF_OK;
}

hf_status hf_get_device_status(void* ws, void* stream, int32_t* site)
{
    if (!ws) return fail(HF_ERR_INVALID_ARG, "ws is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word[2] = {0, 0};
    cudaError_t e = cudaMemcpyAsync(word, ws, sizeof word, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail((int)e, "status read");
    if (word[0] != 0) {
        const uint32_t zero[2] = {0, 0};
        e = cudaMemcpyAsync(ws, zero, sizeof zero, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail((int)e, "status clear");
    }
    if (site) *site = (int32_t)word[1];
    if (word[0] == 0) return HF_OK;
    if (word[0] == HF_DEV_ERR_TIMEOUT)
        return fail(HF_ERR_TIMEOUT, "device wait timed out at site %u", word[1]);
    return fail(HF_ERR_DEVICE_CHECK, "device check failed at site %u (code %u)", word[1], word[0]);
}

hf_status hf_selftest_wait_timeout(void* ws, int32_t limit_us, void* stream)
{
    if (!ws) return fail(HF_ERR_INVALID_ARG, "ws is NULL");
    if (limit_us < 1 || limit_us > 100000) return fail(HF_ERR_INVALID_ARG, "limit_us %d not in [1, 100000]", limit_us);
    HF_LAUNCH(launch_selftest_wait(static_cast<uint32_t*>(ws), (uint64_t)limit_us * 1000ull, stream),
              "self-test launch");
    return HF_OK;
}

}  // extern "C"
