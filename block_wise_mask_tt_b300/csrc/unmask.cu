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

namespace tti {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 4;  // 16-byte loads per thread per batch

struct Red {
    float m;
    float s;
    int a;
};

// Merge two (max, sum of 2^((x - max) * ts), argmax) triples, ts = log2(e) /
// temperature; equal maxima keep the lower id.
__device__ __forceinline__ Red combine(Red x, Red y, float ts) {
    Red r;
    r.m = fmaxf(x.m, y.m);
    if (r.m == -CUDART_INF_F) {
        r.s = 0.f;
        r.a = min(x.a, y.a);
        return r;
    }
    r.s = x.s * exp2f((x.m - r.m) * ts) + y.s * exp2f((y.m - r.m) * ts);
    r.a = (x.m > y.m) ? x.a : (y.m > x.m) ? y.a : min(x.a, y.a);
    return r;
}

__device__ __forceinline__ Red warp_combine(Red v, float ts) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Red w;
        w.m = __shfl_xor_sync(0xffffffffu, v.m, o);
        w.s = __shfl_xor_sync(0xffffffffu, v.s, o);
        w.a = __shfl_xor_sync(0xffffffffu, v.a, o);
        v = combine(v, w, ts);
    }
    return v;
}

// Folds one batch of values (ids ascending in the order given) into the running
// triple of this thread.  The batch maximum comes from a 3-input max tree; its id is
// looked for only when it beats the running maximum (rare once a row's first batches
// are in), and an equal maximum keeps the running, lower id.  The exponentials use one
// packed FMA per pair and a packed running sum.
template <int N>
__device__ __forceinline__ void fold(Red& acc, const float (&x)[N], const int (&id)[N], float ts) {
    static_assert(N % 2 == 0, "pairs");
    float bm = x[0];
#pragma unroll
    for (int i = 1; i + 1 < N; i += 2) bm = ttk::fmax3(bm, x[i], x[i + 1]);
    if (N % 2 == 0) bm = fmaxf(bm, x[N - 1]);
    if (bm > acc.m) {
        int ba = id[N - 1];
#pragma unroll
        for (int i = N - 1; i >= 0; --i)
            if (x[i] == bm) ba = id[i];  // the first (lowest) id attaining the maximum
        acc.s = (acc.m == -CUDART_INF_F) ? 0.f : acc.s * exp2f((acc.m - bm) * ts);
        acc.m = bm;
        acc.a = ba;
    }
    if (acc.m == -CUDART_INF_F) return;
    const float off = -acc.m * ts;
    const uint64_t ts2 = ttk::f2_pack(ts, ts), off2 = ttk::f2_pack(off, off);
    uint64_t s2 = ttk::f2_pack(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        float e0, e1;
        ttk::f2_unpack(ttk::f2_fma(ttk::f2_pack(x[i], x[i + 1]), ts2, off2), e0, e1);
        s2 = ttk::f2_add(s2, ttk::f2_pack(exp2f(e0), exp2f(e1)));
    }
    float s0, s1;
    ttk::f2_unpack(s2, s0, s1);
    acc.s += s0 + s1;
}

// Ticket increment with acquire-release semantics at GPU scope: this thread's earlier
// writes (its partial) are released, and the writes released by the earlier
// increments are acquired by the one that sees the final count.
__device__ __forceinline__ unsigned ticket_add(unsigned* t) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
    return old;
}
// Acquire load of a ticket: every lane of the finishing warp synchronises with all
// the increments before it reads the partials they released.
__device__ __forceinline__ unsigned ticket_acquire(const unsigned* t) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(t) : "memory");
    return v;
}

__device__ __forceinline__ float4 as_f4(Red r) {
    return make_float4(r.m, r.s, __int_as_float(r.a), 0.f);
}
__device__ __forceinline__ Red from_f4(float4 v) { return Red{v.x, v.y, __float_as_int(v.z)}; }

// Warp 0 of the CTA that completed sequence b last: the commit/remask decision for
// its S <= 32 positions, lane = position.
__device__ void decide(const UnmaskParams& p, int b) {
    const int lane = threadIdx.x & 31;
    const int S = p.S;
    const bool in = lane < S;
    const int row = b * S + lane;
    const bool masked = in && __ldcg(p.ids + row) == p.mask_id;
    float conf = 0.f;
    int tok = 0;
    if (masked) {
        const Red r = from_f4(__ldcg(reinterpret_cast<const float4*>(p.row_res) + row));
        conf = (r.s > 0.f) ? 1.0f / r.s : 0.f;
        tok = r.a;
    }
    const unsigned mball = __ballot_sync(0xffffffffu, masked);
    const int m = __popc(mball);
    const int steps_b = __ldcg(p.steps + b);
    bool take = false;
    if (m > 0) {
        // rank = this position's place among the masked ones by confidence (higher
        // first, equal confidences by lower position)
        auto rank_of = [&]() {
            int rank = 0;
            for (int j = 0; j < 32; ++j) {
                const float cj = __shfl_sync(0xffffffffu, conf, j);
                const bool mj = (mball >> j) & 1u;
                rank += (mj && (cj > conf || (cj == conf && j < lane))) ? 1 : 0;
            }
            return rank;
        };
        if (p.mode == 1) {
            // mock-AR: the leftmost masked position
            take = masked && lane == __ffs(mball) - 1;
        } else if (p.mode == 2) {
            // predict-and-noise: the linear schedule leaves floor(S (T - steps - 1) / T)
            // masked; the most confident of the rest are committed (at least one)
            const int left = p.max_steps - steps_b - 1;
            const int keep = (left <= 0) ? 0 : (S * left) / p.max_steps;
            const int k = min(m, max(1, m - keep));
            const int rank = rank_of();
            take = masked && rank < k;
        } else {
            const int left = p.max_steps - steps_b;
            const int k_min = (left > 0) ? (m + left - 1) / left : m;
            const bool above = masked && conf >= p.gamma;
            const unsigned aball = __ballot_sync(0xffffffffu, above);
            if (__popc(aball) >= k_min) {
                take = above;
            } else {
                const int rank = rank_of();
                take = masked && rank < k_min;
            }
        }
    }
    const int n_take = __popc(__ballot_sync(0xffffffffu, take));
    if (in) {
        if (take) {
            p.ids[row] = tok;
            if (p.commit_step) p.commit_step[row] = (uint8_t)(steps_b + 1);
        }
        if (p.commit) p.commit[row] = take ? 1 : 0;
        if (p.conf) p.conf[row] = masked ? conf : 0.f;
    }
    if (lane == 0) {
        if (m > 0) p.steps[b] = steps_b + 1;
        if (p.n_masked) p.n_masked[b] = m - n_take;
        p.ticket[p.B * S + b] = 0u;
    }
}

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
                    for (int e = 0; e < 4; ++e) {
                        id[4 * u + e] = i0 + e;
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
