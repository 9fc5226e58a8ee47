// Host-side interface between the C ABI (tt_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace tti {

// Launches `kernel` so that it may be scheduled while the previous grid in the stream
// is still running (programmatic dependent launch).  Every libtt kernel starts with
// griddepcontrol.wait, so it reads nothing before its predecessor has completed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------------------- adaLN
struct AdalnParams {
    const uint16_t* x;
    const float* shift;
    const float* scale;
    const int32_t* row_index;   // nullable
    int table_rows;
    const int32_t* skip_if_zero;  // nullable: sequences whose entry is 0 are skipped
    uint16_t* y;
    int B, S, H;
    float eps;
    int* err;
};
constexpr int kAdalnMaxH = 8192;
cudaError_t launch_adaln(const AdalnParams& p, cudaStream_t stream);

// ---------------------------------------------------------------------------- logits
struct LogitsParams {
    const int32_t* ids;    // nullable
    const int32_t* steps;  // nullable
    float* logits;
    int B, S, V;
    int32_t mask_id;
    uint32_t seed;
    int block_index;
    int kind;
    float boost_lo, boost_hi;
    const uint32_t* dyn;   // nullable: {seed, block_index} read on the device instead
    int ids_per_cta;       // set by launch_logits
};
cudaError_t launch_logits(const LogitsParams& p, cudaStream_t stream);
cudaError_t launch_set_logits_dyn(uint32_t* dyn, uint32_t seed, int block_index, cudaStream_t stream);

// ---------------------------------------------------------------------------- unmask
struct UnmaskPartial {
    float m;    // max logit of the chunk (mask id excluded)
    float sum;  // sum of exp(logit - m) over the chunk
    int arg;    // lowest id attaining m
    int pad;
};
struct UnmaskParams {
    const float* logits;
    int32_t* ids;
    int32_t* n_masked;   // nullable
    int32_t* steps;
    float* conf;         // nullable
    uint8_t* commit;     // nullable
    uint8_t* commit_step;  // nullable
    int B, S, V;
    int32_t mask_id;
    float gamma;
    int max_steps;
    int mode;           // tt_sampler_kind
    float temp_scale;   // log2(e) / temperature
    int chunk;      // vocabulary entries per CTA (multiple of 1024)
    int n_chunks;
    UnmaskPartial* part;     // [B*S][n_chunks]: one per (row, vocabulary chunk)
    UnmaskPartial* row_res;  // [B*S]: the row's merged (max, sum, argmax)
    unsigned int* ticket;    // [B*S] row tickets then [B] sequence tickets: zero on entry, zero on exit
    int ticket_words;        // B*S + B
    int* err;
};
size_t unmask_workspace_bytes(int B, int S, int V);
void unmask_layout(int B, int S, int V, void* ws, UnmaskParams& p);
cudaError_t launch_unmask(const UnmaskParams& p, cudaStream_t stream);
// Fixed scratch of tt_confidence_unmask_noalloc (a file-scope __device__ array):
// unmask_workspace_bytes(B, S, V) must not exceed this.
constexpr size_t kUnmaskNoallocScratchBytes = size_t(8) << 20;
// Device address of that array on the current device (looked up once per device).
cudaError_t unmask_noalloc_scratch(void** out);

// ------------------------------------------------------------- LM head + unmasking
// The hidden rows of masked positions are gathered into a compact bf16 matrix; a
// persistent tcgen05 GEMM multiplies it with the vocabulary projection W [V][H] and
// reduces every (row, vocabulary chunk) to (max, sum of exponentials, lowest argmax)
// in its epilogue, so no logit is written; a last kernel merges a row's chunks and
// takes the per-sequence decision of the sampler.
constexpr int kLmHeadMaxRows = 4096;  // B * S
struct LmHeadParams {
    const uint16_t* h;     // [B*S][H] bf16 hidden rows
    uint16_t* a_c;         // [B*S][H] masked rows, compacted (workspace)
    int32_t* dest;         // [B*S] compact index of each row, -1 when decoded (workspace)
    int32_t* n_rows;       // number of masked rows (workspace)
    UnmaskPartial* part;   // [B*S][max_chunks] per (compact row, vocabulary chunk) (workspace)
    int rows;              // B * S
    int H, V;
    int n_ctas;            // GEMM grid: one persistent CTA per SM
    UnmaskParams um;       // ids, steps, outputs, sampler, row_res, ticket (decision)
};
struct LmHeadMaps {
    CUtensorMap a;  // A rows: (H, rows) bf16, box 64 x a_rows, 128-B swizzle
    CUtensorMap w;  // W: (H, V) bf16, box 64 x 64, 128-B swizzle
    int a_rows;     // rows of the A box: 128, or the row count rounded up to 8 when below
};
// Rows of the GEMM's A box for a problem of at most `rows` rows: below one 128-row
// tile only the rows that exist are copied.
inline int gemm_a_box_rows(int rows) { return rows >= 128 ? 128 : (rows + 7) / 8 * 8; }
size_t lmhead_a_rows(int rows);  // rows of a_c: B*S rounded up to a multiple of 128
size_t lmhead_workspace_bytes(int B, int S, int H, int n_ctas);
// Fills the workspace pointers of p (p.rows, p.n_ctas set by the caller).
void lmhead_layout(void* ws, LmHeadParams& p);
cudaError_t launch_lmhead(const LmHeadParams& p, const LmHeadMaps& maps, cudaStream_t stream);
cudaError_t lmhead_prepare();  // sets the GEMM's shared-memory limit on this device

// Query/key/value projection of the adaLN output on the same persistent GEMM: y [rows][H]
// times W_qkv [(Hq + 2 Hkv) D][H]^T, rounded to bf16 and stored into q [rows][Hq D],
// k [rows][Hkv D], v [rows][Hkv D].  maps.a covers y (box 64 x 128), maps.w W_qkv.
struct QkvParams {
    uint16_t *q, *k, *v;
    int rows, H, Hq, Hkv, D;
    int n_ctas;
    int* err;
};
cudaError_t launch_qkv(const QkvParams& p, const LmHeadMaps& maps, cudaStream_t stream);

// -------------------------------------------------------------------------- attention
struct AttnGeom {
    int B, S, Hq, Hkv, G, D;
    int R;             // G * S packed query rows per (sequence, kv head), row = s * G + j
    int rows_per_cta;  // rows one split CTA serves: min(R, 256), or 128 on small problems
    int n_rg;          // row groups per (sequence, kv head): ceil(R / rows_per_cta)
    int n_mt;          // 128-row MMA tiles per CTA: ceil(rows_per_cta / 128)
    int max_ctx;       // contiguous: token stride; paged: max_pages * page_size
    int page_size;     // 0 or 64
    int max_pages, num_pages;
    int n_splits;
    int tiles_per_split;  // 128-token tiles per split
    int lpt;              // 1: work units dispatched longest first (ragged paged batches)
    int lpt_dyn;          // lpt: the prep kernel picks the split length per call from the
                          // active sequences (tiles_per_split times 1, 2, 4, ...)
    int fused;            // split row groups are merged inside the split pass (its CTAs
                          // all resident: a cooperative launch), no combine pass
    float scale_log2;     // softmax_scale * log2(e)
};
constexpr int kOrderMaxLen = 1024;       // longest unit (tiles) the longest-first order sorts
constexpr int kOrderMaxUnits = 1 << 20;  // most work units it sorts
bool attn_geometry(int B, int S, int Hq, int Hkv, int D, int max_ctx, int page_size,
                   int max_pages, int num_pages, float softmax_scale, int num_splits,
                   AttnGeom& g, const char** why);
size_t attn_workspace_bytes(const AttnGeom& g);
// Pointers into a workspace of attn_workspace_bytes(g) bytes.  order (lpt only):
// the work units sorted by length, then their count, the split length of the call and
// a flag that is 1 when some row group was split.
void attn_layout(const AttnGeom& g, void* ws, float** part_acc, float** part_ml,
                 unsigned** ticket, int32_t** order);

struct AttnSplitParams {
    AttnGeom g;
    const uint16_t* q;           // bf16 [B][S][Hq][D]
    const int32_t* ctx_len;      // nullable (contiguous only)
    const int32_t* page_table;   // nullable
    const int32_t* skip_if_zero; // nullable
    float* part_acc;             // [B][Hkv][n_splits][R][D]
    float* part_ml;              // [B][Hkv][n_splits][R][2]
    unsigned* ticket;            // fused: [2][B][Hkv][n_rg] arrivals, then finished merges;
                                 // zero on entry and left at zero
    const int32_t* order;        // lpt: [units] work unit of each CTA, then the count
    uint16_t* out;               // bf16 [B][S][Hq][D]: written here by the CTAs of row
                                 // groups with one non-empty split
    float* lse;                  // nullable, [B][S][Hq]: likewise
    int* err;
};
struct AttnMaps {
    CUtensorMap k;   // context keys, bf16 [rows][Hkv][D], box (64, 1, 64), 128-B swizzle
    CUtensorMap v;   // context values
    CUtensorMap kb;  // the block's own keys, bf16 [B*S][Hkv][D], same box
    CUtensorMap vb;  // the block's own values
    // Epilogue stores (128-byte swizzle): the fp32 partial states [splits*B*Hkv][R][D]
    // with box (32, 128, 1), and the bf16 output [B][S][Hq][D] with box
    // (64, G, 128/G, 1) when G divides 128 (out_tma).
    CUtensorMap part;
    CUtensorMap out;
    int out_tma;
};
cudaError_t attn_split_prepare(int D);  // sets the kernel's shared-memory limit on this device
// lpt: sorts the non-empty (row group, split) work units by their number of key tiles,
// longest first, into p.order (one CTA, before the split pass).
cudaError_t launch_attn_order(const AttnSplitParams& p, cudaStream_t stream);
cudaError_t launch_attn_split(const AttnSplitParams& p, const AttnMaps& maps, cudaStream_t stream);

struct AttnMergeParams {
    AttnGeom g;
    const int32_t* order;        // lpt: the prep kernel's output (split length, any split)
    const int32_t* ctx_len;
    const int32_t* skip_if_zero;
    const float* part_acc;
    const float* part_ml;
    uint16_t* out;
    float* lse;
    int* err;
};
cudaError_t launch_attn_merge(const AttnMergeParams& p, cudaStream_t stream);

// ----------------------------------------------------------------------- outer loop
struct AppendParams {
    const uint16_t* k_blk;   // bf16 [B][S][Hkv][D]
    const uint16_t* v_blk;
    uint16_t* k_ctx;         // contiguous [B][capacity][Hkv][D] or pages [P][64][Hkv][D]
    uint16_t* v_ctx;
    const int32_t* page_table;  // [B][max_pages] or null
    int32_t* ctx_len;        // [B] in/out
    const int32_t* ids;      // [B][S] the committed block
    int32_t* generated;      // [B] in/out
    uint8_t* done;           // [B] in/out
    int32_t* out_tokens;     // [B][out_stride] or null: this block at out_offset
    int out_stride, out_offset;
    int B, S, Hkv, D;
    int capacity;            // contiguous: rows per sequence
    int page_size, max_pages, num_pages;
    int32_t eos_id, pad_id;
    int max_new_tokens;
    int* err;
};
cudaError_t launch_append_block(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_block_start(int32_t* ids, int32_t* steps, uint8_t* commit_step, const uint8_t* done,
                               int B, int S, int32_t mask_id, int32_t pad_id, cudaStream_t stream);

// ------------------------------------------------------------------------------ loop
struct InitParams {
    const int32_t* ids;
    int32_t* n_masked;
    uint32_t* iter;   // nullable: loop iteration counter, reset to 0
    int B, S;
    int32_t mask_id;
};
cudaError_t launch_count_masked(const InitParams& p, cudaStream_t stream);

// Sets the block graph's WHILE condition: some sequence still has masked positions
// and steps left, and fewer than max_steps + 1 iterations have run (a hard cap).
struct LoopCondParams {
    const int32_t* n_masked;
    const int32_t* steps;
    uint32_t* iter;
    int B;
    int max_steps;
    unsigned long long handle;
};
cudaError_t launch_loop_cond(const LoopCondParams& p, cudaStream_t stream);

// ------------------------------------------------------------------------- self-test
// One CTA waits on an mbarrier nothing arrives on, for limit_ns, through the bounded
// wait of every kernel; when the wait runs out it sets TT_ERR_TIMEOUT in *err and
// writes 1 to *waited_out (nullable), else 0.
cudaError_t launch_wait_timeout(int* err, unsigned long long limit_ns, int* waited_out,
                                cudaStream_t stream);

}  // namespace tti
