// adaLN prologue: y = LN(x) * (1 + scale(t)) + shift(t), one CTA per (b, s) row.
//
// "Nemotron-Labs-TwoTower" wiki, "Motivation: one network, two roles" and
// "Ablations": the denoiser is conditioned on the diffusion timestep through adaptive
// layer normalization.  LayerNorm over H without learned affine, biased variance,
// fp32 statistics from registers (two passes over the row held in registers), bf16
// output rounded to nearest-even.  The timestep enters only through the modulation
// row: per-sequence vectors, or row row_index[b] of a [rows][H] table (the denoise
// loop passes n_masked, i.e. t = n_masked / S).
#include <cuda_bf16.h>

#include "tt_device.cuh"
#include "tt_internal.h"

namespace tti {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxChunks = kAdalnMaxH / 8 / kThreads;  // 16-byte chunks per thread

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) t += red[i];
    __syncthreads();
    return t;
}

__global__ void __launch_bounds__(kThreads) adaln_kernel(AdalnParams p) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    const int row = blockIdx.x;
    const int b = row / p.S;
    if (p.skip_if_zero != nullptr && __ldg(p.skip_if_zero + b) == 0) return;
    const float* sh;
    const float* sc;
    if (p.row_index != nullptr) {
        const int ri = __ldg(p.row_index + b);
        if (ri < 0 || ri >= p.table_rows) {
            if (threadIdx.x == 0) ttk::report_error(p.err, ttk::kErrDevice);
            return;
        }
        sh = p.shift + (size_t)ri * p.H;
        sc = p.scale + (size_t)ri * p.H;
    } else {
        sh = p.shift + (size_t)b * p.H;
        sc = p.scale + (size_t)b * p.H;
    }
    __shared__ float red[kThreads / 32];
    const int n8 = p.H >> 3;
    // The modulation rows are read only after the two row reductions; pull this
    // thread's part of them into L2 now so that read does not pay the DRAM latency.
    for (int c = threadIdx.x; c < n8; c += kThreads) {
        asm volatile("prefetch.global.L2 [%0];" ::"l"(sh + 8 * c) : "memory");
        asm volatile("prefetch.global.L2 [%0];" ::"l"(sc + 8 * c) : "memory");
    }
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + (size_t)row * p.H);
    float v[kMaxChunks][8];
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxChunks; ++k) {
        const int c = threadIdx.x + k * kThreads;
        if (c < n8) {
            const uint4 u = __ldg(xr + c);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[k][2 * e] = ttk::bf16_bits_to_f32(w[e] & 0xFFFFu);
                v[k][2 * e + 1] = ttk::bf16_bits_to_f32(w[e] >> 16);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) s += v[k][e];
        }
    }
    const float mean = block_sum(s, red) / (float)p.H;
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxChunks; ++k) {
        const int c = threadIdx.x + k * kThreads;
        if (c < n8) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float d = v[k][e] - mean;
                q = fmaf(d, d, q);
            }
        }
    }
    const float var = block_sum(q, red) / (float)p.H;
    const float rstd = 1.0f / sqrtf(var + p.eps);
    uint4* yr = reinterpret_cast<uint4*>(p.y + (size_t)row * p.H);
#pragma unroll
    for (int k = 0; k < kMaxChunks; ++k) {
        const int c = threadIdx.x + k * kThreads;
        if (c < n8) {
            const float4 sh0 = __ldg(reinterpret_cast<const float4*>(sh) + 2 * c);
            const float4 sh1 = __ldg(reinterpret_cast<const float4*>(sh) + 2 * c + 1);
            const float4 sc0 = __ldg(reinterpret_cast<const float4*>(sc) + 2 * c);
            const float4 sc1 = __ldg(reinterpret_cast<const float4*>(sc) + 2 * c + 1);
            const float shv[8] = {sh0.x, sh0.y, sh0.z, sh0.w, sh1.x, sh1.y, sh1.z, sh1.w};
            const float scv[8] = {sc0.x, sc0.y, sc0.z, sc0.w, sc1.x, sc1.y, sc1.z, sc1.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float y0 = fmaf((v[k][2 * e] - mean) * rstd, 1.0f + scv[2 * e], shv[2 * e]);
                const float y1 =
                    fmaf((v[k][2 * e + 1] - mean) * rstd, 1.0f + scv[2 * e + 1], shv[2 * e + 1]);
                const __nv_bfloat162 pr = __floats2bfloat162_rn(y0, y1);
                o[e] = *reinterpret_cast<const uint32_t*>(&pr);
            }
            yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

__global__ void count_masked_kernel(InitParams p) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    const int b = blockIdx.x;
    int n = 0;
    for (int s = threadIdx.x; s < p.S; s += 32) n += (p.ids[b * p.S + s] == p.mask_id) ? 1 : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    if (threadIdx.x == 0) p.n_masked[b] = n;
    if (b == 0 && threadIdx.x == 0 && p.iter != nullptr) *p.iter = 0u;
}

__global__ void loop_cond_kernel(LoopCondParams p) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    int active = 0;
    for (int b = threadIdx.x; b < p.B; b += 32)
        active |= (p.n_masked[b] > 0 && p.steps[b] < p.max_steps) ? 1 : 0;
    active = __any_sync(0xffffffffu, active);
    if (threadIdx.x == 0) {
        const uint32_t it = *p.iter + 1u;
        *p.iter = it;
        const bool go = active && it < (uint32_t)p.max_steps + 1u;
        cudaGraphSetConditional(p.handle, go ? 1u : 0u);
    }
}

}  // namespace

cudaError_t launch_adaln(const AdalnParams& p, cudaStream_t stream) {
    return launch_pdl(adaln_kernel, dim3(p.B * p.S), dim3(kThreads), 0, stream, p);
}

cudaError_t launch_count_masked(const InitParams& p, cudaStream_t stream) {
    return launch_pdl(count_masked_kernel, dim3(p.B), dim3(32), 0, stream, p);
}

cudaError_t launch_loop_cond(const LoopCondParams& p, cudaStream_t stream) {
    return launch_pdl(loop_cond_kernel, dim3(1), dim3(32), 0, stream, p);
}

}  // namespace tti
