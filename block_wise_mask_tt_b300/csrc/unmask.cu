// Confidence unmasking (one denoise step for every sequence of a batch).
//
// "Nemotron-Labs-TwoTower" wiki, "Block-wise generation": each step predicts every
// masked position in parallel, commits those whose confidence clears gamma, keeps a
// floor so the block completes within T steps; the mask token is never emitted and
// decoded positions stay fixed.
//
// Pass structure: a grid of (vocabulary chunk, position, sequence) CTAs streams the
// fp32 logits of masked rows once (16-byte loads that bypass L1, four per thread per
// batch, up to four batches per CTA with six CTAs resident per SM), reducing each chunk
// to (max, lowest argmax, sum of exp).  Completion is
// counted in two levels, so no ticket sees more than max(chunks per row, S) atomic
// increments: the last chunk CTA of a row (acquire-release atomic ticket; nothing
// spins) merges that row's chunk partials into a row result, and the last
// row of a sequence to finish takes the commit/remask decision for its S <= 32
// positions with one warp and applies it in place.
#include <math_constants.h>

#include <mutex>

#include "tt_device.cuh"
#include "tt_internal.h"
#include "unmask_common.cuh"

namespace tti {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 4;  // 16-byte loads per thread per batch

using namespace um;

template <bool kVec>
__global__ void __launch_bounds__(kThreads, 6) unmask_kernel(UnmaskParams p) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    const int c = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
    const int row = b * p.S + s;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    __shared__ Red red[kThreads / 32];

    const bool masked = __ldcg(p.ids + row) == p.mask_id;
    if (masked) {
        const int v0 = c * p.chunk;
        const int v1 = min(p.V, v0 + p.chunk);
        const float* rowp = p.logits + (size_t)row * p.V;
        const int mid = p.mask_id;
        Red acc{-CUDART_INF_F, 0.f, 0x7fffffff};
        if (kVec) {
            // kBatch float4 per thread per batch, ids ascending within the batch.
            const int n4 = (v1 - v0) >> 2;
            const float4* base = reinterpret_cast<const float4*>(rowp + v0);
            int f = tid;
            for (; f + (kBatch - 1) * kThreads < n4; f += kBatch * kThreads) {
                float4 q[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) q[u] = ttk::ld_stream_f4(base + f + u * kThreads);
                float x[4 * kBatch];
                int id[4 * kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int i0 = v0 + 4 * (f + u * kThreads);
                    x[4 * u + 0] = q[u].x;
                    x[4 * u + 1] = q[u].y;
                    x[4 * u + 2] = q[u].z;
                    x[4 * u + 3] = q[u].w;
#pragma unroll
                    for (int e = 0; e < 4; ++e) id[4 * u + e] = i0 + e;
                    // the mask id lies in at most one vector of the row: one test per vector
                    if ((unsigned)(mid - i0) < 4u) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (i0 + e == mid) x[4 * u + e] = -CUDART_INF_F;
                    }
                }
                fold<4 * kBatch>(acc, x, id, p.temp_scale);
            }
            for (; f < n4; f += kThreads) {
                const float4 q = ttk::ld_stream_f4(base + f);
                const int i0 = v0 + 4 * f;
                float x[4] = {q.x, q.y, q.z, q.w};
                int id[4] = {i0, i0 + 1, i0 + 2, i0 + 3};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (id[e] == mid) x[e] = -CUDART_INF_F;
                fold<4>(acc, x, id, p.temp_scale);
            }
        } else {
            for (int v = v0 + tid; v < v1; v += kThreads) {
                float x[2] = {__ldcs(rowp + v), -CUDART_INF_F};
                int id[2] = {v, 0x7fffffff};
                if (v == mid) x[0] = -CUDART_INF_F;
                fold<2>(acc, x, id, p.temp_scale);
            }
        }
        acc = warp_combine(acc, p.temp_scale);
        if (lane == 0) red[warp] = acc;
    }
    __syncthreads();
    if (warp != 0) return;

    // ---- warp 0: chunk partial, then (last chunk of the row) the row result, then
    // (last row of the sequence) the decision.
    if (masked) {
        Red r = (lane < kThreads / 32) ? red[lane] : Red{-CUDART_INF_F, 0.f, 0x7fffffff};
        r = warp_combine(r, p.temp_scale);
        if (lane == 0) __stcg(reinterpret_cast<float4*>(p.part + (size_t)row * p.n_chunks + c), as_f4(r));
    }
    unsigned last_chunk = 0;
    if (lane == 0) last_chunk = (ticket_add(p.ticket + row) == (unsigned)(p.n_chunks - 1)) ? 1u : 0u;
    if (__shfl_sync(0xffffffffu, last_chunk, 0) == 0u) return;
    (void)ticket_acquire(p.ticket + row);
    if (masked) {
        const float4* pp = reinterpret_cast<const float4*>(p.part + (size_t)row * p.n_chunks);
        Red r{-CUDART_INF_F, 0.f, 0x7fffffff};
        for (int cc = lane; cc < p.n_chunks; cc += 32) r = combine(r, from_f4(__ldcg(pp + cc)), p.temp_scale);
        r = warp_combine(r, p.temp_scale);
        if (lane == 0) __stcg(reinterpret_cast<float4*>(p.row_res) + row, as_f4(r));
    }
    __syncwarp();  // every lane's acquire of the row ticket precedes its reset
    unsigned last_row = 0;
    if (lane == 0) {
        p.ticket[row] = 0u;
        last_row = (ticket_add(p.ticket + p.B * p.S + b) == (unsigned)(p.S - 1)) ? 1u : 0u;
    }
    if (__shfl_sync(0xffffffffu, last_row, 0) == 0u) return;
    (void)ticket_acquire(p.ticket + p.B * p.S + b);
    decide(p, b);
}

}  // namespace

size_t unmask_workspace_bytes(int B, int S, int V) {
    // Sized for the smallest chunk (1024 ids), the largest chunk count.
    const size_t rows = (size_t)B * S;
    const int n_chunks = (V + 1023) / 1024;
    size_t part = rows * n_chunks * sizeof(UnmaskPartial);
    part = (part + 255) & ~size_t(255);
    size_t res = rows * sizeof(UnmaskPartial);
    res = (res + 255) & ~size_t(255);
    return part + res + (rows + B + 1) * sizeof(unsigned int);
}

void unmask_layout(int B, int S, int V, void* ws, UnmaskParams& p) {
    // Chunk of 16384 ids (64 KiB of fp32) per CTA, four batches of four 16-byte loads
    // per thread, so the reduction tail is paid once per 64 KiB; fewer rows get
    // smaller chunks so that the grid still covers the SMs several times.
    int chunk = 16384;
    const long long rows = (long long)B * S;
    while (chunk > 2048 && rows * ((V + chunk - 1) / chunk) < 148LL * 3) chunk >>= 1;
    p.chunk = chunk;
    p.n_chunks = (V + chunk - 1) / chunk;
    char* w = reinterpret_cast<char*>(ws);
    size_t part = (size_t)rows * ((V + 1023) / 1024) * sizeof(UnmaskPartial);
    part = (part + 255) & ~size_t(255);
    size_t res = (size_t)rows * sizeof(UnmaskPartial);
    res = (res + 255) & ~size_t(255);
    p.part = reinterpret_cast<UnmaskPartial*>(w);
    p.row_res = reinterpret_cast<UnmaskPartial*>(w + part);
    p.ticket = reinterpret_cast<unsigned int*>(w + part + res);
    p.ticket_words = (int)rows + B;
}

cudaError_t launch_unmask(const UnmaskParams& p, cudaStream_t stream) {
    dim3 grid(p.n_chunks, p.S, p.B);
    if ((p.V & 3) == 0)
        return launch_pdl(unmask_kernel<true>, grid, dim3(kThreads), 0, stream, p);
    else
        return launch_pdl(unmask_kernel<false>, grid, dim3(kThreads), 0, stream, p);
}

}  // namespace tti

namespace tti {

// ---------------------------------------------------------------------------------
// Fixed device scratch for tt_confidence_unmask_noalloc.
//
// Some callers cannot hand the library a workspace: their device memory belongs to
// another allocator, or the calling code may not allocate at all.  For them the
// chunk partials and per-sequence tickets live in this file-scope array instead.
// It is part of the module image, so every device that loads the library holds it
// until the process exits, and every call on a device shares it.
// ---------------------------------------------------------------------------------
namespace {
static __device__ __align__(256) unsigned char g_unmask_noalloc_scratch[kUnmaskNoallocScratchBytes];
}  // namespace

cudaError_t unmask_noalloc_scratch(void** out) {
    // In host code the array's name is only a host-side stand-in; the kernel needs
    // its device address, looked up once per device with that device current.
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_unmask_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace tti
