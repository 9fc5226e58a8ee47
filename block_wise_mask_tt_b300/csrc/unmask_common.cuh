// Confidence-unmasking pieces shared by the unmask kernel and the fused LM-head
// kernels: the (max, sum of exponentials, lowest argmax) reduction, acquire-release
// tickets, and the per-sequence commit/remask decision of every sampler.
//
// "Nemotron-Labs-TwoTower" wiki, "Block-wise generation": commit the positions whose
// confidence clears gamma, with a floor that finishes the block within T steps; the
// mask token is never emitted and decoded positions stay fixed.
#pragma once

#include <math_constants.h>

#include "tt_device.cuh"
#include "tt_internal.h"

namespace tti {
namespace um {
namespace {  // internal linkage in every file that includes this

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
// packed FMA per pair, the SFU's 2^x (relative error about 2^-22, results below 2^-126
// flushed to zero: terms that small cannot move a sum that holds the maximum's 1) and
// a packed running sum.
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
        s2 = ttk::f2_add(s2, ttk::f2_pack(ttk::ex2_ftz(e0), ttk::ex2_ftz(e1)));
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

}  // namespace
}  // namespace um
}  // namespace tti
