/*
 * tt.h - C ABI of libtt: one TwoTower denoiser step over a block of S masked tokens
 * on an NVIDIA B300 (sm_103a).
 *
 * What the operations are (the pages describing the method):
 *   - "Nemotron-Labs-TwoTower" wiki, "Architecture": queries of the noisy block b
 *     attend over the context tower's layer-i KV cache for blocks 0..b-1 followed by
 *     the block's own layer-i keys/values, bidirectionally inside the block.
 *   - same page, "Motivation: one network, two roles" and "Ablations": the denoiser
 *     is conditioned on the diffusion timestep through adaptive LayerNorm (adaLN).
 *   - same page, "Block-wise generation": confidence unmasking - every step predicts
 *     all masked positions, commits those whose confidence clears gamma, keeps a
 *     floor so the block finishes within T steps, never emits the mask token, never
 *     changes decoded positions; the timestep is the fraction still masked.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library never
 *     allocates device memory and never frees anything it was given.  It keeps only
 *     host-side caches (TMA descriptors, instantiated CUDA graphs) keyed by pointers
 *     and shapes.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  Outputs are valid once the stream has synchronised.
 *   - Arguments are validated on the host before anything is launched; an invalid
 *     call returns a status and launches nothing.  Nothing aborts or traps.
 *   - Device-side checks (out-of-range page ids or table rows, bounded waits that
 *     ran out) never fault: the offending work item is skipped and a device error
 *     word is set, which tt_device_status() reads.
 *   - Layouts are dense row-major with the last index fastest.  "bf16" tensors hold
 *     IEEE bfloat16 bit patterns.  Every bf16/fp32 tensor pointer must be 16-byte
 *     aligned.
 *   - Supported shapes: D in {64, 128}; 1 <= S <= 32; Hq % Hkv == 0; G = Hq/Hkv <= 128;
 *     G*S <= 512; H % 8 == 0; V % 4 == 0; page_size 64 when paged.
 */
#ifndef TT_H_
#define TT_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TT_API __attribute__((visibility("default")))
#else
#define TT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* tt_stream_t;

typedef enum {
    TT_OK = 0,
    TT_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or dimension        */
    TT_ERR_UNSUPPORTED = 2,  /* well-formed but outside the supported shapes          */
    TT_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed (see tt_last_error) */
    TT_ERR_DEVICE = 4,       /* device-side range check failed (work item skipped)    */
    TT_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out                    */
    TT_ERR_WORKSPACE = 6     /* workspace pointer null or smaller than required       */
} tt_status;

/* ABI revision of this header. */
#define TT_ABI_VERSION 4
TT_API int tt_abi_version(void);

/* Static name of a status code. */
TT_API const char* tt_status_string(int status);

/* Detail text of the last non-OK status returned on the calling thread ("" if none). */
TT_API const char* tt_last_error(void);

/*
 * Synchronises the current device and reads the device error word that kernels of
 * this library set instead of faulting (TT_ERR_DEVICE or TT_ERR_TIMEOUT, first one
 * wins).  reset != 0 clears it.  Returns TT_OK when no kernel reported a problem.
 */
TT_API tt_status tt_device_status(int reset);

/* --------------------------------------------------------------------------------
 * a1. adaLN prologue
 *
 * "Nemotron-Labs-TwoTower" wiki, "Motivation: one network, two roles": the
 * denoiser is conditioned on the diffusion timestep through adaptive layer
 * normalization (DiT / PixArt-alpha style).  For every row (b, s):
 *     y = (x - mean(x)) / sqrt(var(x) + eps) * (1 + scale) + shift
 * LayerNorm over H with biased variance and no learned affine; fp32 arithmetic,
 * output rounded to nearest-even bf16.
 *
 *   x      bf16 [B][S][H]                         (in)
 *   shift  fp32, scale fp32:                      (in)
 *            row_index == NULL: [B][H], row b for sequence b;
 *            else tables [table_rows][H], row row_index[b] for sequence b
 *            (the denoise loop passes n_masked, i.e. timestep t = n_masked/S).
 *   row_index  int32 [B] or NULL                  (in)
 *   y      bf16 [B][S][H]                         (out; may not alias x)
 * A row_index[b] outside [0, table_rows) skips sequence b and sets TT_ERR_DEVICE.
 * -------------------------------------------------------------------------------- */
TT_API tt_status tt_adaln_modulate(const void* x, const float* shift, const float* scale,
                            const int32_t* row_index, int table_rows, void* y,
                            int B, int S, int H, float eps, tt_stream_t stream);

/* --------------------------------------------------------------------------------
 * a2 + a3. Denoise attention (split-KV pass over the context, then merge + block keys)
 *
 * "Nemotron-Labs-TwoTower" wiki, "Architecture": block queries attend over the
 * concatenation [context-tower layer-i KV cache ; the block's own layer-i K/V],
 * bidirectional inside the block, no causal mask anywhere.  For every (b, s, h):
 *     a_j = softmax_scale * <q[b,s,h,:], key_j>
 *     out[b,s,h,:] = sum_j softmax(a)_j value_j,  lse[b,s,h] = log sum_j exp(a_j)
 * over keys j = context tokens 0..ctx_len[b]-1 of kv head h/G, then block tokens
 * 0..S-1 of kv head h/G.
 *
 *   q            bf16 [B][S][Hq][D]                (in)
 *   k_blk, v_blk bf16 [B][S][Hkv][D]               (in)
 *   contiguous cache (page_size == 0):
 *     k_ctx, v_ctx bf16 [B][max_ctx][Hkv][D]       (in)
 *     page_table   must be NULL
 *   paged cache (page_size == 64):
 *     k_ctx, v_ctx bf16 [num_pages][64][Hkv][D]    (in; the page pool)
 *     page_table   int32 [B][max_pages]            (in; logical page -> pool page)
 *   ctx_len      int32 [B] in [0, max_ctx] (paged: [0, max_pages*64]); NULL means
 *                every sequence has max_ctx tokens (contiguous only).      (in)
 *   out          bf16 [B][S][Hq][D]                (out)
 *   lse          fp32 [B][S][Hq] natural-log sum-exp, or NULL              (out)
 *   workspace    device scratch of tt_denoise_attn_workspace(dims) bytes for the
 *                per-split partial softmax states, two counters per row group (used
 *                when TT_ATTN_FUSED_COMBINE=1 is set in the environment: split CTAs
 *                then merge their row groups themselves; read when a call is
 *                enqueued, so a captured block graph keeps the mode it was captured
 *                with) and, on ragged paged
 *                batches, the order in which the work units run.  Must be
 *                zero-filled before its first use; every call leaves the counters at
 *                zero again.  Calls that share a workspace must not overlap on the
 *                device.
 * A page id outside [0, num_pages) or a ctx_len outside range skips that sequence's
 * context and sets TT_ERR_DEVICE.
 * -------------------------------------------------------------------------------- */
typedef struct {
    int B, S, Hq, Hkv, D;
    int max_ctx;        /* contiguous: token stride of k_ctx/v_ctx; paged: unused       */
    int page_size;      /* 0 = contiguous, 64 = paged                                   */
    int max_pages;      /* paged: columns of page_table                                 */
    int num_pages;      /* paged: pages in the pool                                     */
    float softmax_scale;
    int num_splits;     /* context splits per (sequence, kv head); 0 = library's choice */
} tt_attn_dims;

TT_API size_t tt_denoise_attn_workspace(const tt_attn_dims* dims);

TT_API tt_status tt_denoise_attn(const tt_attn_dims* dims, const void* q, const void* k_blk,
                          const void* v_blk, const void* k_ctx, const void* v_ctx,
                          const int32_t* page_table, const int32_t* ctx_len, void* out,
                          float* lse, void* workspace, size_t workspace_bytes,
                          tt_stream_t stream);

/* --------------------------------------------------------------------------------
 * a4. Synthetic logits (stand-in for the denoiser's LM head, which needs weights)
 *
 * "Nemotron-Labs-TwoTower" wiki, "Block-wise generation": each step predicts all
 * masked positions in parallel.  Row (b, s) of a masked position is regenerated from
 * MurmurHash3_x86_32 (one 4-byte key, 32-bit seed):
 *     h   = m3(s, m3(steps[b], m3(block_index, m3(b, seed))))
 *     r_v = m3(v, h);  z_v = ((sum of the 4 bytes of r_v) - 510) * fp32(1/sqrt(21845))
 *     planted id p = m3(0xFFFFFFFF, h) mod V (p+1 mod V if p == mask_id);
 *     u = (m3(0xFFFFFFFE, h) >> 8) * 2^-24;  kind 0: [lo,hi) = [boost_lo, boost_hi);
 *     kind 1: [0,4) or [10,20) by bit 0 of m3(0xFFFFFFFD, h);
 *     logit_v = z_v, and logit_p = z_p + (lo + u*(hi-lo)), single fp32 roundings.
 *   ids    int32 [B][S] or NULL: when given, only rows with ids == mask_id are written
 *   steps  int32 [B] or NULL (0): the step index entering the hash
 *   logits fp32 [B][S][V] (out)
 * -------------------------------------------------------------------------------- */
typedef struct {
    uint32_t seed;
    int block_index;
    int kind;           /* 0 uniform boost, 1 bimodal boost; in a step, 2 = the LM head */
    float boost_lo, boost_hi;
} tt_logits_spec;

/* logits.kind of a step whose logits come from the LM head (tt_lmhead_unmask) over the
 * step's adaLN output y, with the projection t->w_vocab, instead of the stand-in. */
#define TT_LOGITS_LM_HEAD 2

TT_API tt_status tt_synthetic_logits(const tt_logits_spec* spec, const int32_t* ids,
                              const int32_t* steps, float* logits, int B, int S, int V,
                              int32_t mask_id, tt_stream_t stream);

/* --------------------------------------------------------------------------------
 * a5. Confidence unmasking (one step, every sequence of the batch)
 *
 * "Nemotron-Labs-TwoTower" wiki, "Block-wise generation" (Algorithm 2, confidence
 * unmasking); wispaper summary, "Adaptive Step-wise Generation" (gamma = 0.8 met).
 * For each sequence b with m > 0 positions still masked (ids == mask_id):
 *   per masked position: p = softmax over the vocabulary with the mask id removed;
 *     tok = argmax p (ties to the lowest id); conf = max p;
 *   k_min = ceil(m / (max_steps - steps[b])) (m when no steps are left);
 *   commit {conf >= gamma}, or, when that is fewer than k_min, the k_min most
 *   confident (ties to the lower position); committed positions take tok, the rest
 *   keep mask_id; steps[b] += 1.  Sequences with m == 0 are left untouched.
 *   logits      fp32 [B][S][V]; rows of unmasked positions are not read      (in)
 *   ids         int32 [B][S]                                                 (in/out)
 *   n_masked    int32 [B] positions still masked afterwards, or NULL         (out)
 *   steps       int32 [B]                                                    (in/out)
 *   conf        fp32 [B][S] (0 for positions not masked before), or NULL     (out)
 *   commit      uint8 [B][S] 1 where committed by this call, or NULL         (out)
 *   commit_step uint8 [B][S] set to the new steps[b] where committed, or NULL (in/out)
 *   workspace   tt_confidence_unmask_workspace(B,S,V) bytes; must be zero-filled
 *               before its first use; every call leaves it zero-filled again.
 * Calls that share a workspace must not overlap on the device.
 * -------------------------------------------------------------------------------- */
TT_API size_t tt_confidence_unmask_workspace(int B, int S, int V);

TT_API tt_status tt_confidence_unmask(const float* logits, int32_t* ids, int32_t* n_masked,
                               int32_t* steps, float* conf, uint8_t* commit,
                               uint8_t* commit_step, int B, int S, int V, int32_t mask_id,
                               float gamma, int max_steps, void* workspace,
                               size_t workspace_bytes, tt_stream_t stream);

/* --------------------------------------------------------------------------------
 * Sampler variants of the unmask step
 *
 * "Nemotron-Labs-TwoTower" wiki: "Block-wise generation" names, besides confidence
 * unmasking, the standard predict-and-noise sampler (predict a clean block, re-mask
 * low-confidence positions by the noise schedule); the model-card example in "Release
 * history and artifacts" passes a sampling temperature; the opening summary describes
 * a mock-AR two-tower mode that predicts one token per step.
 *
 * In every mode: the confidence of a masked position is the largest probability of
 * softmax(logits / temperature) with the mask id removed, the token its argmax (ties
 * to the lowest id, independent of the temperature), decoded positions stay fixed,
 * and steps[b] advances by one for every sequence that had a masked position.
 *   TT_SAMPLER_CONFIDENCE: commit every position with confidence >= gamma, and at
 *     least ceil(m / (T - steps)) of them (the most confident) - tt_confidence_unmask
 *     is this mode at temperature 1;
 *   TT_SAMPLER_MOCK_AR: commit exactly one position, the leftmost still masked;
 *   TT_SAMPLER_PREDICT_NOISE: after the step, floor(S * (T - steps - 1) / T)
 *     positions stay masked (0 at the last step), the most confident are committed,
 *     at least one.  Equal confidences go to the lower position.
 * Arguments, layouts, workspace (tt_confidence_unmask_workspace) and errors are those
 * of tt_confidence_unmask; `sampler` is a host pointer.
 * -------------------------------------------------------------------------------- */
typedef enum {
    TT_SAMPLER_CONFIDENCE = 0,
    TT_SAMPLER_MOCK_AR = 1,
    TT_SAMPLER_PREDICT_NOISE = 2
} tt_sampler_kind;

typedef struct {
    int kind;          /* tt_sampler_kind */
    float gamma;       /* confidence threshold (TT_SAMPLER_CONFIDENCE) */
    float temperature; /* > 0 */
    int max_steps;     /* T, 1..255 */
} tt_sampler;

TT_API tt_status tt_sampler_unmask(const float* logits, int32_t* ids, int32_t* n_masked,
                                   int32_t* steps, float* conf, uint8_t* commit,
                                   uint8_t* commit_step, int B, int S, int V, int32_t mask_id,
                                   const tt_sampler* sampler, void* workspace,
                                   size_t workspace_bytes, tt_stream_t stream);

/* --------------------------------------------------------------------------------
 * tt_lmhead_unmask: one sampler step whose logits come from the LM head, fused so
 * that the logits are never written to memory.
 *
 * "Nemotron-Labs-TwoTower" wiki, "Block-wise generation": every step predicts all
 * masked positions of the block and commits the confident ones.  For every masked
 * position (ids[b][s] == mask_id) the logits are
 *     logit[j] = sum_k hidden[b][s][k] * w_vocab[j][k]      (fp32 accumulation)
 * and the step is then exactly that of tt_sampler_unmask on those logits (same
 * confidence, token, tie rules, decision and outputs).  The product runs on the
 * tensor cores and each (row, vocabulary chunk) is reduced to (max, sum of
 * exponentials, lowest argmax) as it leaves the accumulator.
 *
 *   hidden     bf16 [B][S][H], device, 16-byte aligned: the hidden row of every
 *              position (rows of decoded positions are not read)
 *   w_vocab    bf16 [V][H], device, 16-byte aligned: row j projects onto token id j
 *   ids ... commit_step, mask_id, sampler: as tt_sampler_unmask (sampler is a host
 *              pointer)
 *   workspace  tt_lmhead_unmask_workspace(B, S, H) bytes on the current device,
 *              16-byte aligned; its contents on entry do not matter
 * Limits: S <= 32, B*S <= 4096, H a multiple of 8 and >= 64, V >= 64.  Invalid
 * arguments return an error and launch nothing.  Three kernels are launched on
 * `stream`; a wait inside the GEMM that runs out sets the device error word
 * (tt_device_status) instead of hanging.
 * -------------------------------------------------------------------------------- */
TT_API size_t tt_lmhead_unmask_workspace(int B, int S, int H);

TT_API tt_status tt_lmhead_unmask(const void* hidden, const void* w_vocab, int32_t* ids,
                                  int32_t* n_masked, int32_t* steps, float* conf,
                                  uint8_t* commit, uint8_t* commit_step, int B, int S, int H,
                                  int V, int32_t mask_id, const tt_sampler* sampler,
                                  void* workspace, size_t workspace_bytes, tt_stream_t stream);

/* --------------------------------------------------------------------------------
 * tt_qkv_project: the denoiser's query/key/value projection of the adaLN output.
 *
 * "Nemotron-Labs-TwoTower" wiki, "Motivation: one network, two roles" (the denoiser
 * is conditioned on the timestep through adaptive layer normalisation) and
 * "Architecture" (the block's queries and its own keys/values are the denoiser's
 * projections; the block attends over the context cache followed by them).
 *   out[r][c] = sum_k y[r][k] * w_qkv[c][k]   (fp32 accumulation, bf16 RNE store)
 * for r = b*S + s; column c < Hq*D goes to q[b][s][c / D][c % D], the next Hkv*D
 * columns to k_blk, the last Hkv*D to v_blk.
 *   y      bf16 [B][S][H], device, 16-byte aligned
 *   w_qkv  bf16 [(Hq + 2 Hkv) D][H], device, 16-byte aligned
 *   q      bf16 [B][S][Hq][D] (out); k_blk, v_blk bf16 [B][S][Hkv][D] (out)
 * Limits: D in {64, 128}, Hkv divides Hq, H a multiple of 8 and >= 64.  One
 * persistent tcgen05 GEMM kernel on `stream`; no workspace.
 * -------------------------------------------------------------------------------- */
TT_API tt_status tt_qkv_project(const void* y, const void* w_qkv, void* q, void* k_blk, void* v_blk,
                                int B, int S, int H, int Hq, int Hkv, int D, tt_stream_t stream);

/* --------------------------------------------------------------------------------
 * tt_confidence_unmask_noalloc: the same confidence-unmasking step, for callers that
 * cannot provide a workspace.  The pages describing the method have no counterpart
 * to this entry point; it exists for callers whose device memory is owned entirely
 * by another allocator (a serving engine that reserves nearly all HBM up front and
 * hands out only its own buffers) and for code that must not allocate on its hot
 * path (cudaMalloc can synchronise the device and has no latency bound).
 *
 * Arguments, layouts, outputs and errors are those of tt_confidence_unmask without
 * the workspace.  Instead of a workspace it uses a fixed scratch array of 8 MiB
 * (a file-scope __device__ array of the library): every device that loads the
 * library holds those 8 MiB until the process exits.  Sizes whose scratch,
 * tt_confidence_unmask_workspace(B, S, V), exceeds 8 MiB are rejected with
 * TT_ERR_UNSUPPORTED before anything is launched (B*S*ceil(V/1024) up to about
 * 524000, e.g. B*S = 2048 rows at V = 131072 fits).
 *
 * The call allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.  It clears the part of the scratch that must start at zero with
 * cudaMemsetAsync on `stream`, then launches the kernel.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture begins.
 * Every call on a device shares the one array, which keeps the previous call's
 * contents: calls that may overlap on the GPU (other streams, other host threads)
 * race with one another and must be ordered by the caller.
 * -------------------------------------------------------------------------------- */
TT_API tt_status tt_confidence_unmask_noalloc(const float* logits, int32_t* ids,
                                              int32_t* n_masked, int32_t* steps, float* conf,
                                              uint8_t* commit, uint8_t* commit_step, int B,
                                              int S, int V, int32_t mask_id, float gamma,
                                              int max_steps, tt_stream_t stream);

/* --------------------------------------------------------------------------------
 * Self-test of the device-side failure path (no counterpart on the pages: it belongs
 * to this library's error handling, not to the method)
 *
 * Every wait inside the library's kernels (on a TMA copy, a tensor-core operation or
 * another warp) is bounded; a wait that runs out sets TT_ERR_TIMEOUT in the device
 * error word, the kernel drains what it issued and returns, and the context stays
 * usable.  This call exercises exactly that path on purpose: one CTA initialises an
 * mbarrier in shared memory that nothing ever arrives on, waits on it for limit_us
 * microseconds (1 .. 1 000 000) through the same bounded-wait helper, and reports the
 * timeout.  It touches no caller memory, faults nothing and always ends.
 * Afterwards tt_device_status() returns TT_ERR_TIMEOUT (and reset clears it).
 * Errors: TT_ERR_INVALID_ARG for limit_us outside the range; TT_ERR_CUDA if the launch
 * fails.
 * -------------------------------------------------------------------------------- */
TT_API tt_status tt_selftest_wait_timeout(uint32_t limit_us, tt_stream_t stream);

/* --------------------------------------------------------------------------------
 * Whole denoise step and whole block (a1..a5 chained on the device)
 *
 * "Nemotron-Labs-TwoTower" wiki, "Block-wise generation": a block starts fully
 * masked and is refined for up to T steps; the timestep of a step is the fraction
 * still masked, t = n_masked/S, which selects row n_masked of the adaLN tables.
 * One step, for every sequence that still has masked positions:
 *   adaLN(x, table row n_masked[b]) -> y; attention -> attn_out; synthetic logits
 *   for the masked rows (step index steps[b]) -> logits; confidence unmasking.
 * With qkv_proj = 1 the step first projects y into q, k_blk and v_blk
 * (tt_qkv_project with t->w_qkv), so the attention's inputs depend on t.
 * With logits.kind == TT_LOGITS_LM_HEAD the last two are replaced by the fused LM
 * head and sampler step of tt_lmhead_unmask with hidden = y and W = t->w_vocab (no
 * logits buffer is used; H >= 64, V >= 64, B*S <= 4096).
 * Without qkv_proj the adaLN output does not feed the attention: q, k_blk and v_blk
 * are then the caller's fixed tensors (the trained projections are not available).
 * -------------------------------------------------------------------------------- */
typedef struct {
    tt_attn_dims attn;      /* B, S, heads, D, cache layout, softmax scale */
    int H;                  /* adaLN hidden size                           */
    int V;                  /* vocabulary size                             */
    int32_t mask_id;
    float gamma;
    int max_steps;          /* T */
    float ln_eps;
    tt_logits_spec logits;
    int sampler;            /* tt_sampler_kind: TT_SAMPLER_CONFIDENCE (0) for the main sampler */
    float temperature;      /* > 0; 1 = plain softmax */
    int qkv_proj;           /* 1: q, k_blk, v_blk = tt_qkv_project(y, w_qkv) every step */
} tt_step_desc;

typedef struct {
    /* inputs */
    const void* x;              /* bf16 [B][S][H]                           */
    const float* shift_table;   /* fp32 [S+1][H], row n = timestep n/S      */
    const float* scale_table;   /* fp32 [S+1][H]                            */
    const void* q;              /* bf16 [B][S][Hq][D]                       */
    const void* k_blk;          /* bf16 [B][S][Hkv][D]                      */
    const void* v_blk;
    const void* k_ctx;          /* as in tt_denoise_attn                    */
    const void* v_ctx;
    const int32_t* page_table;
    const int32_t* ctx_len;
    /* state, in/out */
    int32_t* ids;               /* int32 [B][S]                             */
    int32_t* n_masked;          /* int32 [B] (step: in/out; loop: out)      */
    int32_t* steps;             /* int32 [B]                                */
    uint8_t* commit_step;       /* uint8 [B][S]                             */
    /* outputs / buffers */
    void* y;                    /* bf16 [B][S][H]: adaLN of the last step   */
    void* attn_out;             /* bf16 [B][S][Hq][D]                       */
    float* logits;              /* fp32 [B][S][V] buffer (NULL with the LM head) */
    float* conf;                /* fp32 [B][S] or NULL                      */
    uint8_t* commit;            /* uint8 [B][S] or NULL                     */
    /* LM head (logits.kind == TT_LOGITS_LM_HEAD), else NULL */
    const void* w_vocab;        /* bf16 [V][H]                              */
    /* projection (qkv_proj == 1), else NULL; q, k_blk, v_blk are then written */
    const void* w_qkv;          /* bf16 [(Hq + 2 Hkv) D][H]                 */
} tt_step_tensors;

/* Workspace for tt_denoise_step / tt_denoise_block_loop (attention partials, unmask
 * partials, tickets).  Must be zero-filled before first use; calls leave it so. */
TT_API size_t tt_denoise_workspace(const tt_step_desc* desc);

/* One step from the given state.  n_masked must equal the count of mask_id in each
 * row of ids (tt_denoise_block_loop establishes it). */
TT_API tt_status tt_denoise_step(const tt_step_desc* desc, const tt_step_tensors* t,
                          void* workspace, size_t workspace_bytes, tt_stream_t stream);

/* Steps until no sequence has masked positions left (at most max_steps - steps[b]
 * per sequence), decided on the device: one launch of a CUDA graph whose
 * conditional WHILE node repeats the step.  n_masked is recomputed from ids first;
 * steps and commit_step continue from their given values (zero them for a fresh
 * block).  The first call with a new set of pointers/shapes builds the graph. */
TT_API tt_status tt_denoise_block_loop(const tt_step_desc* desc, const tt_step_tensors* t,
                                void* workspace, size_t workspace_bytes,
                                tt_stream_t stream);

/* --------------------------------------------------------------------------------
 * Algorithm 1, the block-wise outer loop
 *
 * "Nemotron-Labs-TwoTower" wiki, "Block-wise generation": once a block is clean it is
 * committed, the context tower processes the committed tokens causally to update its
 * caches, and the loop continues with the next block.  The MLX README
 * ("Configuration (diffusion)") adds the stopping knobs: a number of new tokens and an
 * end-of-sequence id.  The context tower's forward needs trained weights: the
 * keys/values appended for a committed block are that block's own k_blk / v_blk.
 * -------------------------------------------------------------------------------- */
typedef struct {
    int32_t eos_id;          /* a block that commits it ends the sequence (-1: none)  */
    int32_t pad_id;          /* fills the positions of finished sequences            */
    int max_new_tokens;      /* a sequence ends once it has generated this many      */
} tt_stop_spec;

/* For every sequence b with done[b] == 0: copies k_blk[b] / v_blk[b] (S rows each) to
 * logical positions ctx_len[b] .. ctx_len[b] + S - 1 of its cache (dims->max_ctx rows
 * per sequence for a contiguous cache, which must fit them; page_table pages for a
 * paged one, which must exist), then ctx_len[b] += S, generated[b] += S, and done[b]
 * = 1 if ids[b] holds stop->eos_id or generated[b] >= stop->max_new_tokens.  A
 * sequence whose rows do not fit is skipped and the device error word set.
 * out_tokens (nullable, int32 [B][out_stride]) receives ids[b] at out_offset, or the
 * pad id for a sequence that was already done.  All pointers are device pointers except
 * dims and stop. */
TT_API tt_status tt_append_block(const tt_attn_dims* dims, const void* k_blk, const void* v_blk,
                                 void* k_ctx, void* v_ctx, const int32_t* page_table,
                                 int32_t* ctx_len, const int32_t* ids, const tt_stop_spec* stop,
                                 int32_t* generated, uint8_t* done, int32_t* out_tokens,
                                 int out_stride, int out_offset, tt_stream_t stream);

/* n_blocks iterations of the outer loop from the current caches: for block k, every
 * running sequence starts fully masked (finished ones hold the pad id), the block is
 * decoded exactly as tt_denoise_block_loop does with logits block index
 * desc->logits.block_index + k, and tt_append_block then appends it (out_offset =
 * k * S).  t->k_ctx, t->v_ctx and t->ctx_len are updated in place (they are in/out
 * here), as are generated and done.  out_tokens: int32 [B][n_blocks * S].  Same
 * workspace as tt_denoise_block_loop; one asynchronous sequence of launches. */
TT_API tt_status tt_generate(const tt_step_desc* desc, const tt_step_tensors* t, int n_blocks,
                             const tt_stop_spec* stop, int32_t* generated, uint8_t* done,
                             int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                             tt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TT_H_ */
