// C ABI of libtt (declared in include/tt.h): argument validation, TMA descriptor
// encoding, kernel launches, and the block loop as a CUDA graph whose WHILE node is
// driven from the device.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include "tt.h"
#include "tt_internal.h"

namespace {

// An NVTX range over one entry point (its validation and enqueue on the host), so that
// a profiler's timeline names every call and step.  With no tool attached the push and
// pop return at once.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
#define TT_RANGE(name) const NvtxRange tt_nvtx_range_(name)

// First error code reported by any libtt kernel on this device (see tt_device_status).
__device__ int g_tt_device_error;

thread_local char g_msg[512] = "";

tt_status fail(tt_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

tt_status cuda_fail(cudaError_t e, const char* what) {
    return fail(TT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define TT_CUDA(call)                                      \
    do {                                                   \
        cudaError_t e_ = (call);                           \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
    } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// exp2 scale of the unmask softmax at temperature tau: log2(e) / tau (exactly the
// plain constant at tau = 1).
float temp_scale(float tau) { return 1.4426950408889634f / tau; }

tt_status need_ptr(const void* p, const char* name, bool align = true) {
    if (p == nullptr) return fail(TT_ERR_INVALID_ARG, "%s is null", name);
    if (align && !aligned16(p)) return fail(TT_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return TT_OK;
}

#define TT_TRY(expr)                      \
    do {                                  \
        tt_status s_ = (expr);            \
        if (s_ != TT_OK) return s_;       \
    } while (0)

// Device address of the error word, looked up once per device.
std::mutex g_mu;
int* g_err_addr[64] = {nullptr};

tt_status device_err_word(int** out) {
    int dev = 0;
    TT_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return fail(TT_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_err_addr[dev] == nullptr) {
        void* p = nullptr;
        TT_CUDA(cudaGetSymbolAddress(&p, g_tt_device_error));
        g_err_addr[dev] = static_cast<int*>(p);
    }
    *out = g_err_addr[dev];
    return TT_OK;
}

// ------------------------------------------------------------------- TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

// Looks the driver's tensor-map encoder up once.  It takes no lock of its own beyond
// the once-flag: the block-graph capture calls it while holding g_mu.
tt_status get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess && fn != nullptr)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (g_encode_err != cudaSuccess) return cuda_fail(g_encode_err, "cudaGetDriverEntryPointByVersion");
    if (g_encode == nullptr) return fail(TT_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    return TT_OK;
}

// bf16 tensor [dim2][dim1][dim0] (dim0 innermost), box (64, box1, box2), 128-B swizzle.
tt_status encode_3d(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1,
                    uint64_t dim2, uint32_t box1, uint32_t box2) {
    TT_TRY(get_encoder());
    const cuuint64_t dims[3] = {dim0, dim1, dim2};
    const cuuint64_t strides[2] = {dim0 * 2, dim0 * dim1 * 2};
    const cuuint32_t box[3] = {64, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(TT_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return TT_OK;
}

// Tensor map of `rank` dimensions (dims[0] innermost; strides in bytes for dims 1..),
// 128-byte swizzle.
tt_status encode_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                     const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
    TT_TRY(get_encoder());
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(map, dtype, rank, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(TT_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return TT_OK;
}

// --------------------------------------------------------------------- validation
tt_status check_attn(const tt_attn_dims* d, tti::AttnGeom& g) {
    if (d == nullptr) return fail(TT_ERR_INVALID_ARG, "dims is null");
    const char* why = nullptr;
    const bool basic_ok = d->B >= 1 && d->S >= 1 && d->Hq >= 1 && d->Hkv >= 1 && d->D >= 1 &&
                          d->Hq % d->Hkv == 0 && d->max_ctx >= 0 && d->num_splits >= 0;
    if (!basic_ok) return fail(TT_ERR_INVALID_ARG, "attention dims out of range");
    if (!tti::attn_geometry(d->B, d->S, d->Hq, d->Hkv, d->D, d->max_ctx, d->page_size, d->max_pages,
                            d->num_pages, d->softmax_scale, d->num_splits, g, &why)) {
        const bool unsupported = strstr(why, "must be at most") || strstr(why, "must be 64 or 128") ||
                                 strstr(why, "page_size");
        return fail(unsupported ? TT_ERR_UNSUPPORTED : TT_ERR_INVALID_ARG, "%s", why);
    }
    return TT_OK;
}

tt_status check_ws(const void* ws, size_t have, size_t need) {
    if (need == 0) return TT_OK;
    if (ws == nullptr) return fail(TT_ERR_WORKSPACE, "workspace is null (need %zu bytes)", need);
    if (!aligned16(ws)) return fail(TT_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
    if (have < need) return fail(TT_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", have, need);
    return TT_OK;
}

struct AttnPlan {
    tti::AttnGeom g;
    tti::AttnMaps maps;
    bool has_ctx;
};

tt_status plan_attn(const tt_attn_dims* d, const void* q, const void* k_blk, const void* v_blk,
                    const void* k_ctx, const void* v_ctx, const int32_t* page_table,
                    const int32_t* ctx_len, const void* out, AttnPlan& pl) {
    TT_TRY(check_attn(d, pl.g));
    TT_TRY(need_ptr(q, "q"));
    TT_TRY(need_ptr(k_blk, "k_blk"));
    TT_TRY(need_ptr(v_blk, "v_blk"));
    TT_TRY(need_ptr(out, "out"));
    const tti::AttnGeom& g = pl.g;
    if (g.page_size) {
        TT_TRY(need_ptr(page_table, "page_table", false));
        TT_TRY(need_ptr(ctx_len, "ctx_len (required with a paged cache)", false));
    } else if (page_table != nullptr) {
        return fail(TT_ERR_INVALID_ARG, "page_table given for a contiguous cache");
    }
    const uint64_t rows = g.page_size ? (uint64_t)g.num_pages * 64u : (uint64_t)g.B * g.max_ctx;
    pl.has_ctx = rows > 0;
    TT_TRY(encode_3d(&pl.maps.kb, k_blk, g.D, g.Hkv, (uint64_t)g.B * g.S, 1, 64));
    TT_TRY(encode_3d(&pl.maps.vb, v_blk, g.D, g.Hkv, (uint64_t)g.B * g.S, 1, 64));
    if (pl.has_ctx) {
        TT_TRY(need_ptr(k_ctx, "k_ctx"));
        TT_TRY(need_ptr(v_ctx, "v_ctx"));
        TT_TRY(encode_3d(&pl.maps.k, k_ctx, g.D, g.Hkv, rows, 1, 64));
        TT_TRY(encode_3d(&pl.maps.v, v_ctx, g.D, g.Hkv, rows, 1, 64));
    } else {
        // No context: the kernel reads only the block's own keys; the context maps are
        // never used, so they are given the block maps.
        pl.maps.k = pl.maps.kb;
        pl.maps.v = pl.maps.vb;
    }
    TT_CUDA(tti::attn_split_prepare(g.D));
    return TT_OK;
}

tt_status sm_count(int* out);

tt_status launch_attention(const AttnPlan& pl, const void* q, const void* k_blk, const void* v_blk,
                           const int32_t* page_table, const int32_t* ctx_len,
                           const int32_t* skip_if_zero, void* out, float* lse, void* ws,
                           int* err, cudaStream_t st) {
    (void)k_blk;
    (void)v_blk;
    tti::AttnGeom g = pl.g;
    if (!pl.has_ctx) {
        g.max_ctx = 0;
        g.page_size = 0;
    }
    float* part_acc = nullptr;
    float* part_ml = nullptr;
    unsigned* ticket = nullptr;
    int32_t* order = nullptr;
    if (!pl.has_ctx) g.lpt = 0;
    // Opt-in (TT_ATTN_FUSED_COMBINE=1 in the environment, read per call): split row
    // groups of a contiguous cache whose whole grid fits one wave (one CTA per SM) are
    // merged inside the split pass, without a combine launch.  Off by default: on the
    // single-sequence and batched workloads the separate combine pass is faster.
    int n_sms = 0;
    TT_TRY(sm_count(&n_sms));
    const char* fz = getenv("TT_ATTN_FUSED_COMBINE");
    const bool fused_on = fz != nullptr && fz[0] == '1' && fz[1] == '\0';
    g.fused = (fused_on && pl.has_ctx && g.page_size == 0 && g.n_splits > 1 && !g.lpt &&
               (long long)g.B * g.Hkv * g.n_rg * g.n_splits <= n_sms) ? 1 : 0;
    tti::attn_layout(g, ws, &part_acc, &part_ml, &ticket, &order);
    // Epilogue store maps: partial states when the context is split and a second pass
    // combines them; the output itself wherever a CTA may write it directly (when G
    // divides 128, so that a 128-row tile covers whole positions).
    tti::AttnMaps maps = pl.maps;
    maps.part = maps.kb;  // placeholders for the maps that are not used
    maps.out = maps.kb;
    maps.out_tma = 0;
    if (g.n_splits > 1) {
        const cuuint64_t dims[3] = {(cuuint64_t)g.D, (cuuint64_t)g.R,
                                    (cuuint64_t)g.B * g.Hkv * g.n_splits};
        const cuuint64_t strides[2] = {(cuuint64_t)g.D * 4, (cuuint64_t)g.R * g.D * 4};
        const cuuint32_t box[3] = {32, 128, 1};
        TT_TRY(encode_map(&maps.part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, part_acc, dims, strides, box));
    }
    if (128 % g.G == 0) {
        const cuuint64_t dims[4] = {(cuuint64_t)g.D, (cuuint64_t)g.Hq, (cuuint64_t)g.S, (cuuint64_t)g.B};
        const cuuint64_t strides[3] = {(cuuint64_t)g.D * 2, (cuuint64_t)g.Hq * g.D * 2,
                                       (cuuint64_t)g.S * g.Hq * g.D * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)g.G, (cuuint32_t)(128 / g.G), 1};
        TT_TRY(encode_map(&maps.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, out, dims, strides, box));
        maps.out_tma = 1;
    }
    tti::AttnSplitParams sp;
    sp.g = g;
    sp.q = static_cast<const uint16_t*>(q);
    sp.ctx_len = pl.has_ctx ? ctx_len : nullptr;
    sp.page_table = pl.has_ctx ? page_table : nullptr;
    sp.skip_if_zero = skip_if_zero;
    sp.part_acc = part_acc;
    sp.part_ml = part_ml;
    sp.ticket = ticket;
    sp.order = order;
    sp.out = static_cast<uint16_t*>(out);
    sp.lse = lse;
    sp.err = err;
    if (order != nullptr) TT_CUDA(tti::launch_attn_order(sp, st));
    TT_CUDA(tti::launch_attn_split(sp, maps, st));
    if (g.n_splits > 1 && !g.fused) {
        tti::AttnMergeParams mp;
        mp.g = g;
        mp.order = order;
        mp.ctx_len = sp.ctx_len;
        mp.skip_if_zero = skip_if_zero;
        mp.part_acc = part_acc;
        mp.part_ml = part_ml;
        mp.out = static_cast<uint16_t*>(out);
        mp.lse = lse;
        mp.err = err;
        TT_CUDA(tti::launch_attn_merge(mp, st));
    }
    return TT_OK;
}

tt_status check_vocab(int B, int S, int V) {
    if (B < 1 || S < 1 || V < 2) return fail(TT_ERR_INVALID_ARG, "B, S must be >= 1 and V >= 2");
    if (S > 32) return fail(TT_ERR_UNSUPPORTED, "S must be at most 32");
    if (V % 4 != 0) return fail(TT_ERR_UNSUPPORTED, "V must be a multiple of 4");
    if ((long long)B * S > 65535LL * 64) return fail(TT_ERR_UNSUPPORTED, "B*S too large");
    return TT_OK;
}

tt_status check_sampler(const tt_sampler* sampler) {
    if (sampler == nullptr) return fail(TT_ERR_INVALID_ARG, "sampler is null");
    if (sampler->kind < TT_SAMPLER_CONFIDENCE || sampler->kind > TT_SAMPLER_PREDICT_NOISE)
        return fail(TT_ERR_INVALID_ARG, "sampler kind must be a tt_sampler_kind");
    if (sampler->max_steps < 1 || sampler->max_steps > 255)
        return fail(TT_ERR_INVALID_ARG, "max_steps must be in [1, 255]");
    if (sampler->gamma != sampler->gamma) return fail(TT_ERR_INVALID_ARG, "gamma is NaN");
    if (!(sampler->temperature > 0.f) || !(sampler->temperature < 1e30f))
        return fail(TT_ERR_INVALID_ARG, "temperature must be positive and finite");
    return TT_OK;
}

// SM count of the current device (one persistent GEMM CTA per SM), cached per device.
tt_status sm_count(int* out) {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    TT_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) {
        *out = cache[dev];
        return TT_OK;
    }
    int n = 0;
    TT_CUDA(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev));
    if (n < 1) return fail(TT_ERR_CUDA, "device reports no SMs");
    if (dev >= 0 && dev < 64) cache[dev] = n;
    *out = n;
    return TT_OK;
}

// The TMA boxes are 64 wide in H and 64 rows of W, so both extents start at 64.
tt_status check_lmhead(int B, int S, int H, int V) {
    if (B < 1 || S < 1) return fail(TT_ERR_INVALID_ARG, "B and S must be >= 1");
    if (S > 32) return fail(TT_ERR_UNSUPPORTED, "S must be at most 32");
    if ((long long)B * S > tti::kLmHeadMaxRows) return fail(TT_ERR_UNSUPPORTED, "B*S must be at most 4096");
    if (H < 64 || H % 8 != 0) return fail(TT_ERR_UNSUPPORTED, "H must be a multiple of 8, at least 64");
    if (V < 64) return fail(TT_ERR_UNSUPPORTED, "V must be at least 64");
    return TT_OK;
}

// The three kernels of the fused LM head + sampler step (arguments already checked).
tt_status enqueue_lmhead(const void* hidden, const void* w_vocab, int32_t* ids, int32_t* n_masked,
                         int32_t* steps, float* conf, uint8_t* commit, uint8_t* commit_step, int B,
                         int S, int H, int V, int32_t mask_id, int kind, float gamma, int max_steps,
                         float temperature, int n_ctas, void* ws, int* err, cudaStream_t st) {
    tti::LmHeadParams p{};
    p.h = static_cast<const uint16_t*>(hidden);
    p.rows = B * S;
    p.H = H;
    p.V = V;
    p.n_ctas = n_ctas;
    tti::UnmaskParams& u = p.um;
    u.logits = nullptr;
    u.ids = ids;
    u.n_masked = n_masked;
    u.steps = steps;
    u.conf = conf;
    u.commit = commit;
    u.commit_step = commit_step;
    u.B = B;
    u.S = S;
    u.V = V;
    u.mask_id = mask_id;
    u.gamma = gamma;
    u.max_steps = max_steps;
    u.mode = kind;
    u.temp_scale = temp_scale(temperature);
    u.chunk = 0;
    u.n_chunks = 0;
    u.err = err;
    tti::lmhead_layout(ws, p);
    tti::LmHeadMaps maps;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)tti::lmhead_a_rows(p.rows)};
        const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
        maps.a_rows = tti::gemm_a_box_rows(p.rows);
        const cuuint32_t box[2] = {64, (cuuint32_t)maps.a_rows};
        TT_TRY(encode_map(&maps.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.a_c, dims, strides, box));
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)V};
        const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
        const cuuint32_t box[2] = {64, 64};
        TT_TRY(encode_map(&maps.w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_vocab, dims, strides, box));
    }
    TT_CUDA(tti::launch_lmhead(p, maps, st));
    return TT_OK;
}

tt_status check_qkv(int B, int S, int H, int Hq, int Hkv, int D) {
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
        return fail(TT_ERR_INVALID_ARG, "B, S, Hq, Hkv must be >= 1 and Hkv must divide Hq");
    if (D != 64 && D != 128) return fail(TT_ERR_UNSUPPORTED, "D must be 64 or 128");
    if (H < 64 || H % 8 != 0) return fail(TT_ERR_UNSUPPORTED, "H must be a multiple of 8, at least 64");
    if ((long long)B * S > 65535LL * 128) return fail(TT_ERR_UNSUPPORTED, "B*S too large");
    return TT_OK;
}

tt_status enqueue_qkv(const void* y, const void* w_qkv, void* q, void* k, void* v, int B, int S, int H,
                      int Hq, int Hkv, int D, int* err, cudaStream_t st) {
    int n_ctas = 0;
    TT_TRY(sm_count(&n_ctas));
    tti::QkvParams p{};
    p.q = static_cast<uint16_t*>(q);
    p.k = static_cast<uint16_t*>(k);
    p.v = static_cast<uint16_t*>(v);
    p.rows = B * S;
    p.H = H;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.D = D;
    p.n_ctas = n_ctas;
    p.err = err;
    tti::LmHeadMaps maps;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)p.rows};
        const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
        maps.a_rows = tti::gemm_a_box_rows(p.rows);
        const cuuint32_t box[2] = {64, (cuuint32_t)maps.a_rows};
        TT_TRY(encode_map(&maps.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, y, dims, strides, box));
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)(Hq + 2 * Hkv) * D};
        const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
        const cuuint32_t box[2] = {64, 64};
        TT_TRY(encode_map(&maps.w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_qkv, dims, strides, box));
    }
    TT_CUDA(tti::launch_qkv(p, maps, st));
    return TT_OK;
}

// ------------------------------------------------------------- step (shared pieces)
struct StepPlan {
    AttnPlan attn;
    size_t attn_ws;
    size_t unmask_ws_off;
    size_t dyn_off;   // {seed, block_index, loop iteration} for the block graph
    size_t total;
    bool lm_head;     // logits from the fused LM head (else the stand-in + unmask)
    int n_ctas;       // LM-head GEMM grid
};

tt_status plan_step(const tt_step_desc* d, StepPlan& sp) {
    if (d == nullptr) return fail(TT_ERR_INVALID_ARG, "desc is null");
    TT_TRY(check_attn(&d->attn, sp.attn.g));
    TT_TRY(check_vocab(d->attn.B, d->attn.S, d->V));
    if (d->H < 8 || d->H % 8 != 0) return fail(TT_ERR_UNSUPPORTED, "H must be a positive multiple of 8");
    if (d->H > tti::kAdalnMaxH) return fail(TT_ERR_UNSUPPORTED, "H must be at most %d", tti::kAdalnMaxH);
    if (d->max_steps < 1 || d->max_steps > 255) return fail(TT_ERR_INVALID_ARG, "max_steps must be in [1, 255]");
    if (d->mask_id < 0 || d->mask_id >= d->V) return fail(TT_ERR_INVALID_ARG, "mask_id outside the vocabulary");
    if (!(d->ln_eps >= 0.f)) return fail(TT_ERR_INVALID_ARG, "ln_eps must be >= 0");
    if (d->logits.kind < 0 || d->logits.kind > TT_LOGITS_LM_HEAD)
        return fail(TT_ERR_INVALID_ARG, "logits.kind must be 0, 1 or TT_LOGITS_LM_HEAD");
    if (d->sampler < TT_SAMPLER_CONFIDENCE || d->sampler > TT_SAMPLER_PREDICT_NOISE)
        return fail(TT_ERR_INVALID_ARG, "sampler must be a tt_sampler_kind");
    if (!(d->temperature > 0.f) || !(d->temperature < 1e30f))
        return fail(TT_ERR_INVALID_ARG, "temperature must be positive and finite");
    if (d->qkv_proj != 0 && d->qkv_proj != 1) return fail(TT_ERR_INVALID_ARG, "qkv_proj must be 0 or 1");
    if (d->qkv_proj)
        TT_TRY(check_qkv(d->attn.B, d->attn.S, d->H, d->attn.Hq, d->attn.Hkv, d->attn.D));
    sp.lm_head = d->logits.kind == TT_LOGITS_LM_HEAD;
    sp.n_ctas = 0;
    size_t tail_ws = 0;
    if (sp.lm_head) {
        TT_TRY(check_lmhead(d->attn.B, d->attn.S, d->H, d->V));
        TT_TRY(sm_count(&sp.n_ctas));
        tail_ws = tti::lmhead_workspace_bytes(d->attn.B, d->attn.S, d->H, sp.n_ctas);
    } else {
        tail_ws = tti::unmask_workspace_bytes(d->attn.B, d->attn.S, d->V);
    }
    sp.attn_ws = (tti::attn_workspace_bytes(sp.attn.g) + 255) & ~size_t(255);
    sp.unmask_ws_off = sp.attn_ws;
    sp.dyn_off = (sp.attn_ws + tail_ws + 255) & ~size_t(255);
    sp.total = sp.dyn_off + 256;
    return TT_OK;
}

tt_status check_step_tensors(const tt_step_desc* d, const tt_step_tensors* t) {
    if (t == nullptr) return fail(TT_ERR_INVALID_ARG, "tensors is null");
    TT_TRY(need_ptr(t->x, "x"));
    TT_TRY(need_ptr(t->shift_table, "shift_table"));
    TT_TRY(need_ptr(t->scale_table, "scale_table"));
    TT_TRY(need_ptr(t->ids, "ids", false));
    TT_TRY(need_ptr(t->n_masked, "n_masked", false));
    TT_TRY(need_ptr(t->steps, "steps", false));
    TT_TRY(need_ptr(t->commit_step, "commit_step", false));
    TT_TRY(need_ptr(t->y, "y"));
    if (d->logits.kind == TT_LOGITS_LM_HEAD) {
        TT_TRY(need_ptr(t->w_vocab, "w_vocab"));
        TT_CUDA(tti::lmhead_prepare());
    } else {
        TT_TRY(need_ptr(t->logits, "logits"));
    }
    if (t->y == t->x) return fail(TT_ERR_INVALID_ARG, "y may not alias x");
    if (d->qkv_proj) {
        TT_TRY(need_ptr(t->w_qkv, "w_qkv"));
        TT_TRY(need_ptr(t->q, "q"));
        TT_TRY(need_ptr(t->k_blk, "k_blk"));
        TT_TRY(need_ptr(t->v_blk, "v_blk"));
        TT_CUDA(tti::lmhead_prepare());
        int n = 0;
        TT_TRY(sm_count(&n));  // cached before any graph capture
    }
    return TT_OK;
}

// cond != 0: enqueued into the block graph, whose logits seed/block index come from
// the workspace slot written before each launch.
tt_status enqueue_step(const tt_step_desc* d, const tt_step_tensors* t, const StepPlan& sp,
                       void* ws, int* err, unsigned long long cond, cudaStream_t st) {
    const int B = d->attn.B, S = d->attn.S;
    tti::AdalnParams ap;
    ap.x = static_cast<const uint16_t*>(t->x);
    ap.shift = t->shift_table;
    ap.scale = t->scale_table;
    ap.row_index = t->n_masked;
    ap.table_rows = S + 1;
    ap.skip_if_zero = t->n_masked;
    ap.y = static_cast<uint16_t*>(t->y);
    ap.B = B;
    ap.S = S;
    ap.H = d->H;
    ap.eps = d->ln_eps;
    ap.err = err;
    TT_CUDA(tti::launch_adaln(ap, st));

    if (d->qkv_proj)  // q, k_blk, v_blk are this step's projections of y
        TT_TRY(enqueue_qkv(t->y, t->w_qkv, const_cast<void*>(t->q), const_cast<void*>(t->k_blk),
                           const_cast<void*>(t->v_blk), B, S, d->H, d->attn.Hq, d->attn.Hkv, d->attn.D,
                           err, st));

    TT_TRY(launch_attention(sp.attn, t->q, t->k_blk, t->v_blk, t->page_table, t->ctx_len,
                            t->n_masked, t->attn_out, nullptr, ws, err, st));

    if (sp.lm_head) {
        TT_TRY(enqueue_lmhead(t->y, t->w_vocab, t->ids, t->n_masked, t->steps, t->conf, t->commit,
                              t->commit_step, B, S, d->H, d->V, d->mask_id, d->sampler, d->gamma,
                              d->max_steps, d->temperature, sp.n_ctas,
                              static_cast<char*>(ws) + sp.unmask_ws_off, err, st));
    } else {
        tti::LogitsParams lp;
        lp.ids = t->ids;
        lp.steps = t->steps;
        lp.logits = t->logits;
        lp.B = B;
        lp.S = S;
        lp.V = d->V;
        lp.mask_id = d->mask_id;
        lp.seed = d->logits.seed;
        lp.block_index = d->logits.block_index;
        lp.kind = d->logits.kind;
        lp.boost_lo = d->logits.boost_lo;
        lp.boost_hi = d->logits.boost_hi;
        lp.dyn = cond ? reinterpret_cast<const uint32_t*>(static_cast<char*>(ws) + sp.dyn_off) : nullptr;
        TT_CUDA(tti::launch_logits(lp, st));

        tti::UnmaskParams up;
        up.logits = t->logits;
        up.ids = t->ids;
        up.n_masked = t->n_masked;
        up.steps = t->steps;
        up.conf = t->conf;
        up.commit = t->commit;
        up.commit_step = t->commit_step;
        up.B = B;
        up.S = S;
        up.V = d->V;
        up.mask_id = d->mask_id;
        up.gamma = d->gamma;
        up.max_steps = d->max_steps;
        up.mode = d->sampler;
        up.temp_scale = temp_scale(d->temperature);
        tti::unmask_layout(B, S, d->V, static_cast<char*>(ws) + sp.unmask_ws_off, up);
        up.err = err;
        TT_CUDA(tti::launch_unmask(up, st));
    }
    if (cond) {
        tti::LoopCondParams lc;
        lc.n_masked = t->n_masked;
        lc.steps = t->steps;
        lc.iter = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + sp.dyn_off) + 2;
        lc.B = B;
        lc.max_steps = d->max_steps;
        lc.handle = cond;
        TT_CUDA(tti::launch_loop_cond(lc, st));
    }
    return TT_OK;
}

// ------------------------------------------------------------------ block graphs
struct GraphKey {
    std::vector<uint64_t> words;
    bool operator<(const GraphKey& o) const { return words < o.words; }
};

struct GraphEntry {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    uint64_t last_use = 0;
};

std::map<GraphKey, GraphEntry> g_graphs;
uint64_t g_graph_clock = 0;
cudaStream_t g_capture_stream[64] = {nullptr};
constexpr size_t kMaxGraphs = 32;

GraphKey make_key(int dev, const tt_step_desc* d_in, const tt_step_tensors* t, const void* ws) {
    GraphKey k;
    k.words.push_back((uint64_t)dev);
    tt_step_desc dc = *d_in;  // seed and block index are read on the device, not baked in
    dc.logits.seed = 0;
    dc.logits.block_index = 0;
    const tt_step_desc* d = &dc;
    const uint64_t* dw = reinterpret_cast<const uint64_t*>(d);
    size_t nd = sizeof(tt_step_desc) / 8;
    for (size_t i = 0; i < nd; ++i) k.words.push_back(dw[i]);
    uint64_t tail = 0;
    std::memcpy(&tail, reinterpret_cast<const char*>(d) + nd * 8, sizeof(tt_step_desc) - nd * 8);
    k.words.push_back(tail);
    const uint64_t* tw = reinterpret_cast<const uint64_t*>(t);
    for (size_t i = 0; i < sizeof(tt_step_tensors) / 8; ++i) k.words.push_back(tw[i]);
    k.words.push_back(reinterpret_cast<uint64_t>(ws));
    return k;
}

void evict_old_graphs() {
    while (g_graphs.size() >= kMaxGraphs) {
        auto oldest = g_graphs.begin();
        for (auto it = g_graphs.begin(); it != g_graphs.end(); ++it)
            if (it->second.last_use < oldest->second.last_use) oldest = it;
        cudaGraphExecDestroy(oldest->second.exec);
        cudaGraphDestroy(oldest->second.graph);
        g_graphs.erase(oldest);
    }
}

tt_status build_block_graph(const tt_step_desc* d, const tt_step_tensors* t, const StepPlan& sp,
                            void* ws, int* err, int dev, GraphEntry& out) {
    if (g_capture_stream[dev] == nullptr)
        TT_CUDA(cudaStreamCreateWithFlags(&g_capture_stream[dev], cudaStreamNonBlocking));
    cudaStream_t cs = g_capture_stream[dev];
    cudaGraph_t graph = nullptr;
    TT_CUDA(cudaGraphCreate(&graph, 0));
    cudaGraphConditionalHandle handle;
    cudaError_t e = cudaGraphConditionalHandleCreate(&handle, graph, 1u, cudaGraphCondAssignDefault);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return cuda_fail(e, "cudaGraphConditionalHandleCreate");
    }
    // init: n_masked from ids
    e = cudaStreamBeginCaptureToGraph(cs, graph, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return cuda_fail(e, "cudaStreamBeginCaptureToGraph");
    }
    tti::InitParams ip{t->ids, t->n_masked,
                       reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + sp.dyn_off) + 2,
                       d->attn.B, d->attn.S, d->mask_id};
    cudaError_t le = tti::launch_count_masked(ip, cs);
    e = cudaStreamEndCapture(cs, &graph);
    if (le != cudaSuccess || e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return cuda_fail(le != cudaSuccess ? le : e, "capturing the loop prologue");
    }
    cudaGraphNode_t init_node = nullptr;
    size_t n_nodes = 1;
    e = cudaGraphGetNodes(graph, &init_node, &n_nodes);
    if (e != cudaSuccess || n_nodes != 1) {
        cudaGraphDestroy(graph);
        return fail(TT_ERR_CUDA, "unexpected prologue graph");
    }
    cudaGraphNodeParams cp = {};
    cp.type = cudaGraphNodeTypeConditional;
    cp.conditional.handle = handle;
    cp.conditional.type = cudaGraphCondTypeWhile;
    cp.conditional.size = 1;
    cudaGraphNode_t cond_node = nullptr;
    e = cudaGraphAddNode(&cond_node, graph, &init_node, nullptr, 1, &cp);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return cuda_fail(e, "cudaGraphAddNode(conditional)");
    }
    cudaGraph_t body = cp.conditional.phGraph_out[0];
    e = cudaStreamBeginCaptureToGraph(cs, body, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return cuda_fail(e, "cudaStreamBeginCaptureToGraph(body)");
    }
    tt_status s = enqueue_step(d, t, sp, ws, err, (unsigned long long)handle, cs);
    cudaGraph_t body_out = body;
    e = cudaStreamEndCapture(cs, &body_out);
    if (s != TT_OK || e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return s != TT_OK ? s : cuda_fail(e, "capturing the loop body");
    }
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return cuda_fail(e, "cudaGraphInstantiate");
    }
    out.graph = graph;
    out.exec = exec;
    return TT_OK;
}


}  // namespace

// =================================================================================
// exported
// =================================================================================
extern "C" {

int tt_abi_version(void) { return TT_ABI_VERSION; }

const char* tt_status_string(int s) {
    switch (s) {
        case TT_OK: return "TT_OK";
        case TT_ERR_INVALID_ARG: return "TT_ERR_INVALID_ARG";
        case TT_ERR_UNSUPPORTED: return "TT_ERR_UNSUPPORTED";
        case TT_ERR_CUDA: return "TT_ERR_CUDA";
        case TT_ERR_DEVICE: return "TT_ERR_DEVICE";
        case TT_ERR_TIMEOUT: return "TT_ERR_TIMEOUT";
        case TT_ERR_WORKSPACE: return "TT_ERR_WORKSPACE";
        default: return "TT_ERR_UNKNOWN";
    }
}

const char* tt_last_error(void) { return g_msg; }

tt_status tt_device_status(int reset) {
    int* addr = nullptr;
    TT_TRY(device_err_word(&addr));
    TT_CUDA(cudaDeviceSynchronize());
    int code = 0;
    TT_CUDA(cudaMemcpy(&code, addr, sizeof(int), cudaMemcpyDeviceToHost));
    if (reset && code != 0) {
        const int zero = 0;
        TT_CUDA(cudaMemcpy(addr, &zero, sizeof(int), cudaMemcpyHostToDevice));
    }
    if (code == 0) return TT_OK;
    if (code == TT_ERR_TIMEOUT) return fail(TT_ERR_TIMEOUT, "a bounded device wait ran out");
    return fail(TT_ERR_DEVICE, "a device-side range check failed (code %d)", code);
}

tt_status tt_adaln_modulate(const void* x, const float* shift, const float* scale,
                            const int32_t* row_index, int table_rows, void* y, int B, int S, int H,
                            float eps, tt_stream_t stream) {
    TT_RANGE("tt_adaln_modulate");
    if (B < 1 || S < 1 || H < 1) return fail(TT_ERR_INVALID_ARG, "B, S, H must be positive");
    if (H % 8 != 0) return fail(TT_ERR_UNSUPPORTED, "H must be a multiple of 8");
    if (H > tti::kAdalnMaxH) return fail(TT_ERR_UNSUPPORTED, "H must be at most %d", tti::kAdalnMaxH);
    if ((long long)B * S > 0x7fffffffLL) return fail(TT_ERR_UNSUPPORTED, "B*S too large");
    if (!(eps >= 0.f)) return fail(TT_ERR_INVALID_ARG, "eps must be >= 0");
    TT_TRY(need_ptr(x, "x"));
    TT_TRY(need_ptr(shift, "shift"));
    TT_TRY(need_ptr(scale, "scale"));
    TT_TRY(need_ptr(y, "y"));
    if (x == y) return fail(TT_ERR_INVALID_ARG, "y may not alias x");
    if (row_index != nullptr && table_rows < 1) return fail(TT_ERR_INVALID_ARG, "table_rows must be >= 1");
    int* err = nullptr;
    TT_TRY(device_err_word(&err));
    tti::AdalnParams p;
    p.x = static_cast<const uint16_t*>(x);
    p.shift = shift;
    p.scale = scale;
    p.row_index = row_index;
    p.table_rows = table_rows;
    p.skip_if_zero = nullptr;
    p.y = static_cast<uint16_t*>(y);
    p.B = B;
    p.S = S;
    p.H = H;
    p.eps = eps;
    p.err = err;
    TT_CUDA(tti::launch_adaln(p, reinterpret_cast<cudaStream_t>(stream)));
    return TT_OK;
}

size_t tt_denoise_attn_workspace(const tt_attn_dims* dims) {
    tti::AttnGeom g;
    if (check_attn(dims, g) != TT_OK) return 0;
    return tti::attn_workspace_bytes(g);
}

tt_status tt_denoise_attn(const tt_attn_dims* dims, const void* q, const void* k_blk,
                          const void* v_blk, const void* k_ctx, const void* v_ctx,
                          const int32_t* page_table, const int32_t* ctx_len, void* out, float* lse,
                          void* workspace, size_t workspace_bytes, tt_stream_t stream) {
    TT_RANGE("tt_denoise_attn");
    AttnPlan pl;
    TT_TRY(plan_attn(dims, q, k_blk, v_blk, k_ctx, v_ctx, page_table, ctx_len, out, pl));
    if (lse != nullptr) TT_TRY(need_ptr(lse, "lse", false));
    TT_TRY(check_ws(workspace, workspace_bytes, tti::attn_workspace_bytes(pl.g)));
    int* err = nullptr;
    TT_TRY(device_err_word(&err));
    return launch_attention(pl, q, k_blk, v_blk, page_table, ctx_len, nullptr, out, lse, workspace,
                            err, reinterpret_cast<cudaStream_t>(stream));
}

tt_status tt_synthetic_logits(const tt_logits_spec* spec, const int32_t* ids, const int32_t* steps,
                              float* logits, int B, int S, int V, int32_t mask_id,
                              tt_stream_t stream) {
    TT_RANGE("tt_synthetic_logits");
    if (spec == nullptr) return fail(TT_ERR_INVALID_ARG, "spec is null");
    TT_TRY(check_vocab(B, S, V));
    if (spec->kind != 0 && spec->kind != 1) return fail(TT_ERR_INVALID_ARG, "kind must be 0 or 1");
    TT_TRY(need_ptr(logits, "logits"));
    tti::LogitsParams p;
    p.ids = ids;
    p.steps = steps;
    p.logits = logits;
    p.B = B;
    p.S = S;
    p.V = V;
    p.mask_id = mask_id;
    p.seed = spec->seed;
    p.block_index = spec->block_index;
    p.kind = spec->kind;
    p.boost_lo = spec->boost_lo;
    p.boost_hi = spec->boost_hi;
    p.dyn = nullptr;
    TT_CUDA(tti::launch_logits(p, reinterpret_cast<cudaStream_t>(stream)));
    return TT_OK;
}

size_t tt_confidence_unmask_workspace(int B, int S, int V) {
    if (check_vocab(B, S, V) != TT_OK) return 0;
    return tti::unmask_workspace_bytes(B, S, V);
}

tt_status tt_confidence_unmask(const float* logits, int32_t* ids, int32_t* n_masked, int32_t* steps,
                               float* conf, uint8_t* commit, uint8_t* commit_step, int B, int S,
                               int V, int32_t mask_id, float gamma, int max_steps, void* workspace,
                               size_t workspace_bytes, tt_stream_t stream) {
    TT_RANGE("tt_confidence_unmask");
    TT_TRY(check_vocab(B, S, V));
    if (mask_id < 0 || mask_id >= V) return fail(TT_ERR_INVALID_ARG, "mask_id outside the vocabulary");
    if (max_steps < 1 || max_steps > 255) return fail(TT_ERR_INVALID_ARG, "max_steps must be in [1, 255]");
    if (gamma != gamma) return fail(TT_ERR_INVALID_ARG, "gamma is NaN");
    TT_TRY(need_ptr(logits, "logits"));
    TT_TRY(need_ptr(ids, "ids", false));
    TT_TRY(need_ptr(steps, "steps", false));
    TT_TRY(check_ws(workspace, workspace_bytes, tti::unmask_workspace_bytes(B, S, V)));
    int* err = nullptr;
    TT_TRY(device_err_word(&err));
    tti::UnmaskParams p;
    p.logits = logits;
    p.ids = ids;
    p.n_masked = n_masked;
    p.steps = steps;
    p.conf = conf;
    p.commit = commit;
    p.commit_step = commit_step;
    p.B = B;
    p.S = S;
    p.V = V;
    p.mask_id = mask_id;
    p.gamma = gamma;
    p.max_steps = max_steps;
    p.mode = TT_SAMPLER_CONFIDENCE;
    p.temp_scale = temp_scale(1.0f);
    tti::unmask_layout(B, S, V, workspace, p);
    p.err = err;
    TT_CUDA(tti::launch_unmask(p, reinterpret_cast<cudaStream_t>(stream)));
    return TT_OK;
}

tt_status tt_sampler_unmask(const float* logits, int32_t* ids, int32_t* n_masked, int32_t* steps,
                            float* conf, uint8_t* commit, uint8_t* commit_step, int B, int S, int V,
                            int32_t mask_id, const tt_sampler* sampler, void* workspace,
                            size_t workspace_bytes, tt_stream_t stream) {
    TT_RANGE("tt_sampler_unmask");
    TT_TRY(check_sampler(sampler));
    TT_TRY(check_vocab(B, S, V));
    if (mask_id < 0 || mask_id >= V) return fail(TT_ERR_INVALID_ARG, "mask_id outside the vocabulary");
    TT_TRY(need_ptr(logits, "logits"));
    TT_TRY(need_ptr(ids, "ids", false));
    TT_TRY(need_ptr(steps, "steps", false));
    TT_TRY(check_ws(workspace, workspace_bytes, tti::unmask_workspace_bytes(B, S, V)));
    int* err = nullptr;
    TT_TRY(device_err_word(&err));
    tti::UnmaskParams p;
    p.logits = logits;
    p.ids = ids;
    p.n_masked = n_masked;
    p.steps = steps;
    p.conf = conf;
    p.commit = commit;
    p.commit_step = commit_step;
    p.B = B;
    p.S = S;
    p.V = V;
    p.mask_id = mask_id;
    p.gamma = sampler->gamma;
    p.max_steps = sampler->max_steps;
    p.mode = sampler->kind;
    p.temp_scale = temp_scale(sampler->temperature);
    tti::unmask_layout(B, S, V, workspace, p);
    p.err = err;
    TT_CUDA(tti::launch_unmask(p, reinterpret_cast<cudaStream_t>(stream)));
    return TT_OK;
}

tt_status tt_confidence_unmask_noalloc(const float* logits, int32_t* ids, int32_t* n_masked,
                                       int32_t* steps, float* conf, uint8_t* commit,
                                       uint8_t* commit_step, int B, int S, int V, int32_t mask_id,
                                       float gamma, int max_steps, tt_stream_t stream) {
    TT_RANGE("tt_confidence_unmask_noalloc");
    TT_TRY(check_vocab(B, S, V));
    if (mask_id < 0 || mask_id >= V) return fail(TT_ERR_INVALID_ARG, "mask_id outside the vocabulary");
    if (max_steps < 1 || max_steps > 255) return fail(TT_ERR_INVALID_ARG, "max_steps must be in [1, 255]");
    if (gamma != gamma) return fail(TT_ERR_INVALID_ARG, "gamma is NaN");
    TT_TRY(need_ptr(logits, "logits"));
    TT_TRY(need_ptr(ids, "ids", false));
    TT_TRY(need_ptr(steps, "steps", false));
    const size_t need = tti::unmask_workspace_bytes(B, S, V);
    if (need > tti::kUnmaskNoallocScratchBytes)
        return fail(TT_ERR_UNSUPPORTED,
                    "B=%d, S=%d, V=%d needs %zu bytes of scratch; the fixed scratch of "
                    "tt_confidence_unmask_noalloc holds %zu (use tt_confidence_unmask with a workspace)",
                    B, S, V, need, tti::kUnmaskNoallocScratchBytes);
    int* err = nullptr;
    TT_TRY(device_err_word(&err));
    void* scratch = nullptr;
    TT_CUDA(tti::unmask_noalloc_scratch(&scratch));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    tti::UnmaskParams p;
    p.logits = logits;
    p.ids = ids;
    p.n_masked = n_masked;
    p.steps = steps;
    p.conf = conf;
    p.commit = commit;
    p.commit_step = commit_step;
    p.B = B;
    p.S = S;
    p.V = V;
    p.mask_id = mask_id;
    p.gamma = gamma;
    p.max_steps = max_steps;
    p.mode = TT_SAMPLER_CONFIDENCE;
    p.temp_scale = temp_scale(1.0f);
    tti::unmask_layout(B, S, V, scratch, p);
    p.err = err;
    // The array keeps whatever the previous call left; the tickets must start at zero.
    TT_CUDA(cudaMemsetAsync(p.ticket, 0, (size_t)p.ticket_words * sizeof(unsigned int), st));
    TT_CUDA(tti::launch_unmask(p, st));
    return TT_OK;
}

size_t tt_denoise_workspace(const tt_step_desc* desc) {
    StepPlan sp;
    if (plan_step(desc, sp) != TT_OK) return 0;
    return sp.total;
}

tt_status tt_denoise_step(const tt_step_desc* desc, const tt_step_tensors* t, void* workspace,
                          size_t workspace_bytes, tt_stream_t stream) {
    TT_RANGE("tt_denoise_step");
    StepPlan sp;
    TT_TRY(plan_step(desc, sp));
    TT_TRY(check_step_tensors(desc, t));
    TT_TRY(plan_attn(&desc->attn, t->q, t->k_blk, t->v_blk, t->k_ctx, t->v_ctx, t->page_table,
                     t->ctx_len, t->attn_out, sp.attn));
    TT_TRY(check_ws(workspace, workspace_bytes, sp.total));
    int* err = nullptr;
    TT_TRY(device_err_word(&err));
    return enqueue_step(desc, t, sp, workspace, err, 0ull, reinterpret_cast<cudaStream_t>(stream));
}

tt_status tt_denoise_block_loop(const tt_step_desc* desc, const tt_step_tensors* t, void* workspace,
                                size_t workspace_bytes, tt_stream_t stream) {
    TT_RANGE("tt_denoise_block_loop");
    StepPlan sp;
    TT_TRY(plan_step(desc, sp));
    TT_TRY(check_step_tensors(desc, t));
    TT_TRY(plan_attn(&desc->attn, t->q, t->k_blk, t->v_blk, t->k_ctx, t->v_ctx, t->page_table,
                     t->ctx_len, t->attn_out, sp.attn));
    TT_TRY(check_ws(workspace, workspace_bytes, sp.total));
    int* err = nullptr;
    TT_TRY(device_err_word(&err));
    int dev = 0;
    TT_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return fail(TT_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    const GraphKey key = make_key(dev, desc, t, workspace);
    auto it = g_graphs.find(key);
    if (it == g_graphs.end()) {
        evict_old_graphs();
        GraphEntry ge;
        TT_TRY(build_block_graph(desc, t, sp, workspace, err, dev, ge));
        it = g_graphs.emplace(key, ge).first;
    }
    it->second.last_use = ++g_graph_clock;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    TT_CUDA(tti::launch_set_logits_dyn(
        reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + sp.dyn_off), desc->logits.seed,
        desc->logits.block_index, st));
    TT_CUDA(cudaGraphLaunch(it->second.exec, st));
    return TT_OK;
}

tt_status tt_append_block(const tt_attn_dims* dims, const void* k_blk, const void* v_blk,
                          void* k_ctx, void* v_ctx, const int32_t* page_table, int32_t* ctx_len,
                          const int32_t* ids, const tt_stop_spec* stop, int32_t* generated,
                          uint8_t* done, int32_t* out_tokens, int out_stride, int out_offset,
                          tt_stream_t stream) {
    TT_RANGE("tt_append_block");
    tti::AttnGeom g;
    TT_TRY(check_attn(dims, g));
    if (stop == nullptr) return fail(TT_ERR_INVALID_ARG, "stop is null");
    TT_TRY(need_ptr(k_blk, "k_blk"));
    TT_TRY(need_ptr(v_blk, "v_blk"));
    TT_TRY(need_ptr(k_ctx, "k_ctx"));
    TT_TRY(need_ptr(v_ctx, "v_ctx"));
    TT_TRY(need_ptr(ctx_len, "ctx_len", false));
    TT_TRY(need_ptr(ids, "ids", false));
    TT_TRY(need_ptr(generated, "generated", false));
    TT_TRY(need_ptr(done, "done", false));
    if (g.page_size) TT_TRY(need_ptr(page_table, "page_table", false));
    else if (g.max_ctx < g.S) return fail(TT_ERR_INVALID_ARG, "a contiguous cache needs max_ctx >= S");
    if (out_tokens != nullptr && (out_offset < 0 || out_stride < out_offset + g.S))
        return fail(TT_ERR_INVALID_ARG, "out_tokens must hold S tokens at out_offset");
    int* err = nullptr;
    TT_TRY(device_err_word(&err));
    tti::AppendParams p;
    p.k_blk = static_cast<const uint16_t*>(k_blk);
    p.v_blk = static_cast<const uint16_t*>(v_blk);
    p.k_ctx = static_cast<uint16_t*>(k_ctx);
    p.v_ctx = static_cast<uint16_t*>(v_ctx);
    p.page_table = g.page_size ? page_table : nullptr;
    p.ctx_len = ctx_len;
    p.ids = ids;
    p.generated = generated;
    p.done = done;
    p.out_tokens = out_tokens;
    p.out_stride = out_stride;
    p.out_offset = out_offset;
    p.B = g.B;
    p.S = g.S;
    p.Hkv = g.Hkv;
    p.D = g.D;
    p.capacity = g.page_size ? 0 : g.max_ctx;
    p.page_size = g.page_size;
    p.max_pages = g.max_pages;
    p.num_pages = g.num_pages;
    p.eos_id = stop->eos_id;
    p.pad_id = stop->pad_id;
    p.max_new_tokens = stop->max_new_tokens;
    p.err = err;
    TT_CUDA(tti::launch_append_block(p, reinterpret_cast<cudaStream_t>(stream)));
    return TT_OK;
}

tt_status tt_generate(const tt_step_desc* desc, const tt_step_tensors* t, int n_blocks,
                      const tt_stop_spec* stop, int32_t* generated, uint8_t* done,
                      int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                      tt_stream_t stream) {
    TT_RANGE("tt_generate");
    if (desc == nullptr || t == nullptr || stop == nullptr)
        return fail(TT_ERR_INVALID_ARG, "desc, tensors and stop must be given");
    if (n_blocks < 1) return fail(TT_ERR_INVALID_ARG, "n_blocks must be >= 1");
    if ((long long)n_blocks * desc->attn.S > 0x7fffffffLL) return fail(TT_ERR_INVALID_ARG, "n_blocks too large");
    TT_TRY(need_ptr(t->ctx_len, "ctx_len (in/out here)", false));
    TT_TRY(need_ptr(out_tokens, "out_tokens", false));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int B = desc->attn.B, S = desc->attn.S;
    for (int k = 0; k < n_blocks; ++k) {
        TT_CUDA(tti::launch_block_start(t->ids, t->steps, t->commit_step, done, B, S, desc->mask_id,
                                        stop->pad_id, st));
        tt_step_desc dk = *desc;
        dk.logits.block_index = desc->logits.block_index + k;
        TT_TRY(tt_denoise_block_loop(&dk, t, workspace, workspace_bytes, stream));
        TT_TRY(tt_append_block(&desc->attn, t->k_blk, t->v_blk, const_cast<void*>(t->k_ctx),
                               const_cast<void*>(t->v_ctx), t->page_table,
                               const_cast<int32_t*>(t->ctx_len), t->ids, stop, generated, done,
                               out_tokens, n_blocks * S, k * S, stream));
    }
    return TT_OK;
}

size_t tt_lmhead_unmask_workspace(int B, int S, int H) {
    if (check_lmhead(B, S, H, 64) != TT_OK) return 0;
    int n = 0;
    if (sm_count(&n) != TT_OK) return 0;
    return tti::lmhead_workspace_bytes(B, S, H, n);
}

tt_status tt_lmhead_unmask(const void* hidden, const void* w_vocab, int32_t* ids, int32_t* n_masked,
                           int32_t* steps, float* conf, uint8_t* commit, uint8_t* commit_step, int B,
                           int S, int H, int V, int32_t mask_id, const tt_sampler* sampler,
                           void* workspace, size_t workspace_bytes, tt_stream_t stream) {
    TT_RANGE("tt_lmhead_unmask");
    TT_TRY(check_lmhead(B, S, H, V));
    TT_TRY(check_sampler(sampler));
    if (mask_id < 0 || mask_id >= V) return fail(TT_ERR_INVALID_ARG, "mask_id outside the vocabulary");
    TT_TRY(need_ptr(hidden, "hidden"));
    TT_TRY(need_ptr(w_vocab, "w_vocab"));
    TT_TRY(need_ptr(ids, "ids", false));
    TT_TRY(need_ptr(steps, "steps", false));
    int n_ctas = 0;
    TT_TRY(sm_count(&n_ctas));
    TT_TRY(check_ws(workspace, workspace_bytes, tti::lmhead_workspace_bytes(B, S, H, n_ctas)));
    int* err = nullptr;
    TT_TRY(device_err_word(&err));
    return enqueue_lmhead(hidden, w_vocab, ids, n_masked, steps, conf, commit, commit_step, B, S, H, V,
                          mask_id, sampler->kind, sampler->gamma, sampler->max_steps, sampler->temperature,
                          n_ctas, workspace, err, reinterpret_cast<cudaStream_t>(stream));
}

tt_status tt_qkv_project(const void* y, const void* w_qkv, void* q, void* k_blk, void* v_blk, int B, int S,
                         int H, int Hq, int Hkv, int D, tt_stream_t stream) {
    TT_RANGE("tt_qkv_project");
    TT_TRY(check_qkv(B, S, H, Hq, Hkv, D));
    TT_TRY(need_ptr(y, "y"));
    TT_TRY(need_ptr(w_qkv, "w_qkv"));
    TT_TRY(need_ptr(q, "q"));
    TT_TRY(need_ptr(k_blk, "k_blk"));
    TT_TRY(need_ptr(v_blk, "v_blk"));
    int* err = nullptr;
    TT_TRY(device_err_word(&err));
    return enqueue_qkv(y, w_qkv, q, k_blk, v_blk, B, S, H, Hq, Hkv, D, err, reinterpret_cast<cudaStream_t>(stream));
}

tt_status tt_selftest_wait_timeout(uint32_t limit_us, tt_stream_t stream) {
    TT_RANGE("tt_selftest_wait_timeout");
    if (limit_us < 1 || limit_us > 1000000u)
        return fail(TT_ERR_INVALID_ARG, "limit_us must be in [1, 1000000]");
    int* err = nullptr;
    TT_TRY(device_err_word(&err));
    TT_CUDA(tti::launch_wait_timeout(err, 1000ull * limit_us, nullptr, reinterpret_cast<cudaStream_t>(stream)));
    return TT_OK;
}

}  // extern "C"
