// Synthetic per-step logits: the stand-in for the denoiser's LM head.
//
// "Nemotron-Labs-TwoTower" wiki, "Block-wise generation": every denoising step
// predicts all masked positions in parallel.  Trained LM-head weights are not
// available, so each masked row is regenerated from a counter-based hash,
// MurmurHash3_x86_32 of one 4-byte key (Austin Appleby's published definition):
//   h   = m3(s, m3(step, m3(block, m3(b, seed))))
//   z_v = (byte-sum of m3(v, h) - 510) * fp32(1/sqrt(21845))   (Irwin-Hall(4) noise)
//   the planted id m3(~0, h) mod V (stepped past the mask id) gets lo + u*(hi-lo),
//   u = (m3(~1, h) >> 8) * 2^-24, [lo, hi) chosen by the kind (bimodal: bit 0 of
//   m3(~2, h) picks [0,4) or [10,20)).
// Every float operation is a single correctly rounded fp32 op (no contraction), so
// the values are bit-identical to any other IEEE implementation of the same recipe.
#include "tt_device.cuh"
#include "tt_internal.h"

namespace tti {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxIdsPerCta = 8192;
constexpr int kRows = 4;  // positions of one sequence per CTA

__device__ __forceinline__ uint32_t m3(uint32_t key, uint32_t seed) {
    uint32_t k = key * 0xCC9E2D51u;
    k = __funnelshift_l(k, k, 15);
    k *= 0x1B873593u;
    uint32_t h = seed ^ k;
    h = __funnelshift_l(h, h, 13);
    h = h * 5u + 0xE6546B64u;
    h ^= 4u;  // key length in bytes
    h ^= h >> 16;
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    h ^= h >> 16;
    return h;
}

// The hash of id v under a row's seed h0, split so that the work on the key alone is
// shared by every row: with k' = rotl(v * c1, 15) * c2 the mixing step is
// rotl(h0 ^ k', 13) = rotl(h0, 13) ^ rotl(k', 13) (a rotation distributes over xor), so
// key_part(v) = rotl(k', 13) is computed once per id and seed_part(h0) = rotl(h0, 13)
// once per row.  The length xor (h ^= 4, then h ^= h >> 16) is taken as
// h ^ (h >> 16) ^ 4, since the 4 does not reach the shifted bits.  Exact in 32-bit
// arithmetic: the same value as m3(v, h0).
__device__ __forceinline__ uint32_t key_part(uint32_t k_premul) {
    uint32_t k = __funnelshift_l(k_premul, k_premul, 15);
    k *= 0x1B873593u;
    return __funnelshift_l(k, k, 13);
}
__device__ __forceinline__ uint32_t seed_part(uint32_t h0) { return __funnelshift_l(h0, h0, 13); }
__device__ __forceinline__ uint32_t m3_split(uint32_t key, uint32_t seed) {
    uint32_t h = seed ^ key;
    h = h * 5u + 0xE6546B64u;
    h = h ^ (h >> 16) ^ 4u;
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    h ^= h >> 16;
    return h;
}

__device__ __forceinline__ float noise(uint32_t r) {
    // sum of the four bytes minus 510, the offset taken as the dot product's addend
    const int sum = (int)__dp4a(r, 0x01010101u, (uint32_t)-510);
    // fp32(1/sqrt(4*(256^2-1)/12)) = 0x3BDDB446
    return __fmul_rn(__int2float_rn(sum), __uint_as_float(0x3BDDB446u));
}

// One CTA: a chunk of ids_per_cta ids of kRows consecutive positions of one sequence.
// The per-id key work is shared by the CTA's masked rows.
__global__ void __launch_bounds__(kThreads) logits_kernel(LogitsParams p) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    const int c = blockIdx.x, s0 = blockIdx.y * kRows, b = blockIdx.z;
    const uint32_t step = p.steps ? (uint32_t)__ldg(p.steps + b) : 0u;
    const uint32_t seed = p.dyn ? p.dyn[0] : p.seed;
    const uint32_t block = p.dyn ? p.dyn[1] : (uint32_t)p.block_index;
    // Row r's hash chain and planted id, computed by thread r and shared
    __shared__ uint32_t s_hs[kRows], s_planted[kRows];
    __shared__ float s_boost[kRows];
    __shared__ int s_act[kRows];
    if (threadIdx.x < kRows) {
        const int r = threadIdx.x, s = s0 + r;
        uint32_t h = m3((uint32_t)b, seed);
        h = m3(block, h);
        h = m3(step, h);
        h = m3((uint32_t)s, h);
        s_act[r] = (s < p.S && (p.ids == nullptr || __ldg(p.ids + b * p.S + s) == p.mask_id)) ? 1 : 0;
        s_hs[r] = seed_part(h);
        uint32_t pl = m3(0xFFFFFFFFu, h) % (uint32_t)p.V;
        if ((int)pl == p.mask_id) pl = (pl + 1u) % (uint32_t)p.V;
        s_planted[r] = pl;
        const float u = __fmul_rn((float)(m3(0xFFFFFFFEu, h) >> 8), 5.9604644775390625e-08f);
        float lo = p.boost_lo, hi = p.boost_hi;
        if (p.kind == 1) {
            const bool upper = (m3(0xFFFFFFFDu, h) & 1u) != 0u;
            lo = upper ? 10.0f : 0.0f;
            hi = upper ? 20.0f : 4.0f;
        }
        s_boost[r] = __fadd_rn(lo, __fmul_rn(u, __fsub_rn(hi, lo)));
    }
    __syncthreads();
    bool act[kRows];
    uint32_t hs[kRows], planted[kRows];
    float boost[kRows];
    bool any = false;
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        act[r] = s_act[r] != 0;
        any |= act[r];
        hs[r] = s_hs[r];
        planted[r] = s_planted[r];
        boost[r] = s_boost[r];
    }
    if (!any) return;

    float* rows = p.logits + (size_t)(b * p.S + s0) * p.V;
    const int v0 = c * p.ids_per_cta;
    const int v1 = min(p.V, v0 + p.ids_per_cta);
    constexpr uint32_t kC1 = 0xCC9E2D51u;
    if ((p.V & 3) == 0) {
        for (int v = v0 + 4 * threadIdx.x; v < v1; v += 4 * kThreads) {
            const uint32_t k0 = (uint32_t)v * kC1;
            const uint32_t kp[4] = {key_part(k0), key_part(k0 + kC1), key_part(k0 + 2u * kC1),
                                    key_part(k0 + 3u * kC1)};
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                if (!act[r]) continue;
                float o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) o[e] = noise(m3_split(kp[e], hs[r]));
                const unsigned d = planted[r] - (uint32_t)v;
                if (d < 4u) {  // the planted id is in this group of four
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (d == (unsigned)e) o[e] = __fadd_rn(o[e], boost[r]);
                }
                *reinterpret_cast<float4*>(rows + (size_t)r * p.V + v) = make_float4(o[0], o[1], o[2], o[3]);
            }
        }
    } else {
        for (int v = v0 + threadIdx.x; v < v1; v += kThreads) {
            const uint32_t kp = key_part((uint32_t)v * kC1);
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                if (!act[r]) continue;
                float z = noise(m3_split(kp, hs[r]));
                if (v == (int)planted[r]) z = __fadd_rn(z, boost[r]);
                rows[(size_t)r * p.V + v] = z;
            }
        }
    }
}

__global__ void set_dyn_kernel(uint32_t* dyn, uint32_t seed, uint32_t block) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    dyn[0] = seed;
    dyn[1] = block;
}

}  // namespace

cudaError_t launch_set_logits_dyn(uint32_t* dyn, uint32_t seed, int block_index, cudaStream_t stream) {
    return launch_pdl(set_dyn_kernel, dim3(1), dim3(1), 0, stream, dyn, seed, (uint32_t)block_index);
}

cudaError_t launch_logits(const LogitsParams& p_in, cudaStream_t stream) {
    // 8192 ids per CTA; small batches take smaller chunks (down to 1024) so that the
    // grid still covers every SM about twice
    LogitsParams p = p_in;
    const long long groups = (long long)((p.S + kRows - 1) / kRows) * p.B;
    p.ids_per_cta = kMaxIdsPerCta;
    while (p.ids_per_cta > 1024 && groups * ((p.V + p.ids_per_cta - 1) / p.ids_per_cta) < 2LL * 148)
        p.ids_per_cta >>= 1;
    dim3 grid((p.V + p.ids_per_cta - 1) / p.ids_per_cta, (p.S + kRows - 1) / kRows, p.B);
    return launch_pdl(logits_kernel, grid, dim3(kThreads), 0, stream, p);
}

}  // namespace tti
