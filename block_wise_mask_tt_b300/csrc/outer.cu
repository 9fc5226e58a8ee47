// Algorithm 1, the block-wise outer loop: once a block is committed, its keys/values
// join the context cache and the next block starts.
//
// "Nemotron-Labs-TwoTower" wiki, "Block-wise generation": the context tower processes
// each committed block causally to update its caches, and the loop continues with the
// next block.  The context tower's forward needs trained weights; the keys/values it
// would append are stood in for by the block's own keys/values.  The MLX port's
// README ("Configuration (diffusion)") adds the stopping knobs: a number of new tokens
// and an end-of-sequence id.
//
// append_block_kernel, one CTA per sequence: checks that the S new rows fit (capacity
// of a contiguous cache, or existing pages of a paged one), copies the block's K and V
// rows to logical positions ctx_len .. ctx_len + S - 1 with 16-byte loads and stores,
// records the block's tokens, then advances ctx_len / generated and sets done on the
// end-of-sequence id or the length limit.  A sequence already done is left alone.
#include "tt_device.cuh"
#include "tt_internal.h"

namespace tti {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) append_block_kernel(AppendParams p) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const int S = p.S;
    const bool was_done = p.done[b] != 0;
    // The block's tokens go to the output (pad for a sequence that is already done).
    if (p.out_tokens != nullptr)
        for (int s = tid; s < S; s += kThreads)
            p.out_tokens[(size_t)b * p.out_stride + p.out_offset + s] = was_done ? p.pad_id : p.ids[b * S + s];
    if (was_done) return;
    const int ctx = p.ctx_len[b];
    // Where the new rows go: every one must exist, else nothing is written.
    int bad = 0;
    if (p.page_size) {
        const int pg0 = ctx / 64, pg1 = (ctx + S - 1) / 64;
        for (int pg = pg0 + tid; pg <= pg1; pg += kThreads) {
            const int id = (pg < p.max_pages) ? p.page_table[(size_t)b * p.max_pages + pg] : -1;
            bad |= (id < 0 || id >= p.num_pages) ? 1 : 0;
        }
    } else {
        bad = (ctx < 0 || ctx + S > p.capacity) ? 1 : 0;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) ttk::report_error(p.err, ttk::kErrDevice);
        return;
    }
    const int vec = p.D / 8;  // 16-byte vectors per (token, kv head) row
    const int n = S * p.Hkv * vec;
    for (int i = tid; i < n; i += kThreads) {
        const int c = i % vec;
        const int h = (i / vec) % p.Hkv;
        const int s = i / (vec * p.Hkv);
        const int pos = ctx + s;
        const size_t src = (((size_t)b * S + s) * p.Hkv + h) * p.D;
        const size_t row = p.page_size ? (size_t)p.page_table[(size_t)b * p.max_pages + pos / 64] * 64 + pos % 64
                                       : (size_t)b * p.capacity + pos;
        const size_t dst = (row * p.Hkv + h) * p.D;
        reinterpret_cast<uint4*>(p.k_ctx + dst)[c] = reinterpret_cast<const uint4*>(p.k_blk + src)[c];
        reinterpret_cast<uint4*>(p.v_ctx + dst)[c] = reinterpret_cast<const uint4*>(p.v_blk + src)[c];
    }
    int eos = 0;
    for (int s = tid; s < S; s += kThreads) eos |= (p.ids[b * S + s] == p.eos_id) ? 1 : 0;
    eos = __syncthreads_or(eos);
    if (tid == 0) {
        p.ctx_len[b] = ctx + S;
        const int gen = p.generated[b] + S;
        p.generated[b] = gen;
        if (eos || gen >= p.max_new_tokens) p.done[b] = 1;
    }
}

// Start of a block: positions of running sequences are masked, those of finished
// sequences hold the pad id (so every step skips them); steps and commit steps reset.
__global__ void block_start_kernel(int32_t* ids, int32_t* steps, uint8_t* commit_step,
                                   const uint8_t* done, int B, int S, int32_t mask_id, int32_t pad_id) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= B * S) return;
    const int b = i / S;
    ids[i] = done[b] ? pad_id : mask_id;
    commit_step[i] = 0;
    if (i % S == 0) steps[b] = 0;
}

}  // namespace

cudaError_t launch_append_block(const AppendParams& p, cudaStream_t stream) {
    return launch_pdl(append_block_kernel, dim3(p.B), dim3(kThreads), 0, stream, p);
}

cudaError_t launch_block_start(int32_t* ids, int32_t* steps, uint8_t* commit_step, const uint8_t* done,
                               int B, int S, int32_t mask_id, int32_t pad_id, cudaStream_t stream) {
    const int n = B * S;
    return launch_pdl(block_start_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, ids, steps,
                      commit_step, done, B, S, mask_id, pad_id);
}

}  // namespace tti
