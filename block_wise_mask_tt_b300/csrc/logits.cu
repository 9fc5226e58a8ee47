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
constexpr int kIdsPerCta = 8192;

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

// MurmurHash3_x86_32 of a 4-byte key whose first multiplication (key * c1) has
// already been done: the vocabulary loop advances k by c1 per id instead of
// multiplying (exact in 32-bit arithmetic).
__device__ __forceinline__ uint32_t m3_premul(uint32_t k, uint32_t seed) {
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

__device__ __forceinline__ float noise(uint32_t r) {
    const int sum = (int)__dp4a(r, 0x01010101u, 0u);  // sum of the four bytes
    // fp32(1/sqrt(4*(256^2-1)/12)) = 0x3BDDB446
    return __fmul_rn(__int2float_rn(sum - 510), __uint_as_float(0x3BDDB446u));
}

__global__ void __launch_bounds__(kThreads) logits_kernel(LogitsParams p) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    const int c = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
    const int row = b * p.S + s;
    if (p.ids != nullptr && __ldg(p.ids + row) != p.mask_id) return;
    const uint32_t step = p.steps ? (uint32_t)__ldg(p.steps + b) : 0u;
    const uint32_t seed = p.dyn ? p.dyn[0] : p.seed;
    const uint32_t block = p.dyn ? p.dyn[1] : (uint32_t)p.block_index;
    uint32_t h = m3((uint32_t)b, seed);
    h = m3(block, h);
    h = m3(step, h);
    h = m3((uint32_t)s, h);
    uint32_t planted = m3(0xFFFFFFFFu, h) % (uint32_t)p.V;
    if ((int)planted == p.mask_id) planted = (planted + 1u) % (uint32_t)p.V;
    const float u = __fmul_rn((float)(m3(0xFFFFFFFEu, h) >> 8), 5.9604644775390625e-08f);
    float lo = p.boost_lo, hi = p.boost_hi;
    if (p.kind == 1) {
        const bool upper = (m3(0xFFFFFFFDu, h) & 1u) != 0u;
        lo = upper ? 10.0f : 0.0f;
        hi = upper ? 20.0f : 4.0f;
    }
    const float boost = __fadd_rn(lo, __fmul_rn(u, __fsub_rn(hi, lo)));

    float* rowp = p.logits + (size_t)row * p.V;
    const int v0 = c * kIdsPerCta;
    const int v1 = min(p.V, v0 + kIdsPerCta);
    if ((p.V & 3) == 0) {
        constexpr uint32_t kC1 = 0xCC9E2D51u;
        for (int v = v0 + 4 * threadIdx.x; v < v1; v += 4 * kThreads) {
            const uint32_t k0 = (uint32_t)v * kC1;
            float4 o;
            o.x = noise(m3_premul(k0, h));
            o.y = noise(m3_premul(k0 + kC1, h));
            o.z = noise(m3_premul(k0 + 2u * kC1, h));
            o.w = noise(m3_premul(k0 + 3u * kC1, h));
            const unsigned d = planted - (uint32_t)v;
            if (d < 4u) {  // the planted id is in this group of four
                if (d == 0) o.x = __fadd_rn(o.x, boost);
                if (d == 1) o.y = __fadd_rn(o.y, boost);
                if (d == 2) o.z = __fadd_rn(o.z, boost);
                if (d == 3) o.w = __fadd_rn(o.w, boost);
            }
            *reinterpret_cast<float4*>(rowp + v) = o;
        }
    } else {
        for (int v = v0 + threadIdx.x; v < v1; v += kThreads) {
            float z = noise(m3((uint32_t)v, h));
            if (v == (int)planted) z = __fadd_rn(z, boost);
            rowp[v] = z;
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

cudaError_t launch_logits(const LogitsParams& p, cudaStream_t stream) {
    dim3 grid((p.V + kIdsPerCta - 1) / kIdsPerCta, p.S, p.B);
    return launch_pdl(logits_kernel, grid, dim3(kThreads), 0, stream, p);
}

}  // namespace tti
