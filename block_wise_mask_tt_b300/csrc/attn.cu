// Denoise attention: split-KV pass over the context cache on tcgen05, then a merge
// pass that also folds in the block's own (bidirectional) keys.
//
// "Nemotron-Labs-TwoTower" wiki, "Architecture": block queries attend over the
// context tower's layer-i KV cache followed by the denoiser's own layer-i keys and
// values for the block, with bidirectional attention inside the block.
//
// Split pass, one CTA per (context split, 128-row tile, kv head, sequence):
//   * rows of the tile are the packed (block position s, query head j of the GQA
//     group) pairs, row = s*G + j, so one kv head's K/V tile serves G*S query rows
//     and QK^T / PV are real dense contractions (M = 128, N = 64 keys, K = D);
//   * Q (loaded once) and 64-token K/V tiles are staged in shared memory by TMA with
//     128-byte swizzle; K/V use a 2-stage ring so the next tile streams in while the
//     current one is processed;
//   * S = Q K^T is accumulated in tensor memory (TMEM), read back one row per
//     thread, turned into P = exp2(S*scale*log2e - m) with an online max that is
//     only raised (and O rescaled in TMEM) when it grows by more than 2^8;
//   * P (bf16) goes to shared memory in the canonical K-major swizzled layout and
//     O += P V is accumulated in TMEM (V as an MN-major operand, no transpose);
//   * the tile's (m, l, O) partial state goes to the workspace.
// Merge pass, one CTA per (block position, kv head, sequence), one warp per query
// head: combines the partial states of the splits and the S block keys.
#include <math_constants.h>

#include "tt_device.cuh"
#include "tt_internal.h"

namespace tti {
namespace {

constexpr int kSplitThreads = 128;
constexpr int kTileKeys = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct SplitSmem {
    static constexpr int NP = D / 64;                    // 64-element (128 B) column parts
    static constexpr uint32_t kQPart = 128 * 128;        // 128 rows x 128 B
    static constexpr uint32_t kKVPart = kTileKeys * 128; // 64 rows x 128 B
    static constexpr uint32_t kStage = NP * kKVPart;
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + NP * kQPart;
    static constexpr uint32_t kV = kK + 2 * kStage;
    static constexpr uint32_t kP = kV + 2 * kStage;
    static constexpr uint32_t kBar = kP + 128 * 128;
    static constexpr uint32_t kEnd = kBar + 64;
    static constexpr uint32_t kBytes = kEnd + 1024;       // alignment slack
    static constexpr uint32_t kTmemCols = (D == 128) ? 256 : 128;
    static constexpr uint32_t kOCol = (D == 128) ? 128 : 64;
};

__device__ __forceinline__ void tie32(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31]));
}

template <int D>
__global__ void __launch_bounds__(kSplitThreads, 2)
    attn_split_kernel(const __grid_constant__ AttnSplitParams p,
                      const __grid_constant__ CUtensorMap tmq,
                      const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
    using L = SplitSmem<D>;
    constexpr int NP = L::NP;
    constexpr uint32_t kIdescQK = ttk::idesc_bf16(128, kTileKeys, false, false);
    constexpr uint32_t kIdescPV = ttk::idesc_bf16(128, D, false, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + 48);
    volatile int* sh_flag = reinterpret_cast<volatile int*>(smem + L::kBar + 56);

    const AttnGeom& g = p.g;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int split = blockIdx.x;
    const int gkv = blockIdx.y / g.n_row_tiles;
    const int rt = blockIdx.y % g.n_row_tiles;
    const int b = blockIdx.z;

    if (p.skip_if_zero != nullptr && __ldg(p.skip_if_zero + b) == 0) return;
    const int cap = g.page_size ? g.max_pages * g.page_size : g.max_ctx;
    const int ctx = p.ctx_len ? __ldg(p.ctx_len + b) : g.max_ctx;
    if (ctx < 0 || ctx > cap) {
        if (tid == 0 && split == 0 && blockIdx.y == 0) ttk::report_error(p.err, ttk::kErrDevice);
        return;
    }
    const int n_tiles = (ctx + kTileKeys - 1) / kTileKeys;
    const int t0 = split * g.tiles_per_split;
    const int t1 = min(n_tiles, t0 + g.tiles_per_split);
    if (t0 >= t1) return;  // this split is empty; the merge pass does not read it
    const int nt = t1 - t0;

    const int row_local = tid;  // TMEM lane == tile row == thread
    const int r_global = rt * g.rows_per_tile + row_local;
    const bool row_valid = row_local < g.rows_per_tile && r_global < g.R;
    const size_t pidx =
        ((size_t)(b * g.Hkv + gkv) * g.n_splits + split) * (size_t)g.R + (size_t)r_global;

    if (g.page_size) {
        int bad = 0;
        for (int t = t0 + tid; t < t1; t += kSplitThreads) {
            const int pg = __ldg(p.page_table + (size_t)b * g.max_pages + t);
            bad |= (pg < 0 || pg >= g.num_pages) ? 1 : 0;
        }
        if (__syncthreads_or(bad)) {
            if (tid == 0) ttk::report_error(p.err, ttk::kErrDevice);
            if (row_valid) {
                p.part_ml[2 * pidx + 0] = -CUDART_INF_F;
                p.part_ml[2 * pidx + 1] = 0.f;
            }
            return;
        }
    }

    const uint32_t sQ = ttk::smem_u32(smem + L::kQ);
    const uint32_t sK = ttk::smem_u32(smem + L::kK);
    const uint32_t sV = ttk::smem_u32(smem + L::kV);
    const uint32_t sP = ttk::smem_u32(smem + L::kP);
    const uint32_t bar_q = ttk::smem_u32(&bars[0]);
    const uint32_t bar_full0 = ttk::smem_u32(&bars[1]);
    const uint32_t bar_mma = ttk::smem_u32(&bars[3]);

    if (warp == 0) {
        ttk::tmem_alloc(ttk::smem_u32(tmem_slot), L::kTmemCols);
        ttk::tmem_relinquish();
    }
    if (tid == 0) {
        ttk::mbar_init(bar_q, 1);
        ttk::mbar_init(bar_full0, 1);
        ttk::mbar_init(bar_full0 + 8, 1);
        ttk::mbar_init(bar_mma, 1);
        ttk::fence_mbar_init();
    }
    // Rows past the packed (s, head) rows of this tile are zero so they stay finite.
    if (row_local >= g.rows_per_tile) {
#pragma unroll
        for (int part = 0; part < NP; ++part) {
            uint4* dst = reinterpret_cast<uint4*>(smem + L::kQ + part * L::kQPart + row_local * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    ttk::fence_proxy_async_smem();
    ttk::tc_fence_before();
    __syncthreads();
    ttk::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem;
    const uint32_t tO = tmem + L::kOCol;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

    auto kv_row = [&](int t) -> int {
        if (g.page_size) return __ldg(p.page_table + (size_t)b * g.max_pages + t) * kTileKeys;
        return b * g.max_ctx + t * kTileKeys;
    };
    auto issue_kv = [&](int stage, int t) {
        const uint32_t fb = bar_full0 + 8u * (uint32_t)stage;
        const int row0 = kv_row(t);
        ttk::mbar_arrive_expect_tx(fb, 2u * L::kStage);
#pragma unroll
        for (int part = 0; part < NP; ++part) {
            ttk::tma_load_3d(sK + stage * L::kStage + part * L::kKVPart, &tmk, part * 64, gkv, row0, fb);
            ttk::tma_load_3d(sV + stage * L::kStage + part * L::kKVPart, &tmv, part * 64, gkv, row0, fb);
        }
    };

    if (tid == 0) {
        ttk::mbar_arrive_expect_tx(bar_q, (uint32_t)(NP * g.rows_per_tile * 128));
#pragma unroll
        for (int part = 0; part < NP; ++part)
            ttk::tma_load_3d(sQ + part * L::kQPart, &tmq, part * 64, gkv * g.G,
                             b * g.S + rt * g.s_per_tile, bar_q);
        issue_kv(0, t0);
    }

    float m_run = -CUDART_INF_F;
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
        const int stage = j & 1;
        const int t = t0 + j;
        // ---- S = Q K^T (one thread issues; everyone else waits at the CTA barrier)
        if (tid == 0) {
            if (j + 1 < nt) issue_kv(stage ^ 1, t + 1);
            bool w = (j > 0) || ttk::mbar_wait(bar_q, 0);
            w = w && ttk::mbar_wait(bar_full0 + 8u * (uint32_t)stage, (uint32_t)((j >> 1) & 1));
            if (w) {
                ttk::tc_fence_after();
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t koff = (uint32_t)(k & 3) * 32u;
                    const uint64_t a = ttk::sdesc_sw128(sQ + (k >> 2) * L::kQPart + koff, 16, 1024);
                    const uint64_t bd =
                        ttk::sdesc_sw128(sK + stage * L::kStage + (k >> 2) * L::kKVPart + koff, 16, 1024);
                    ttk::mma_bf16_ss(tS, a, bd, kIdescQK, k > 0 ? 1u : 0u);
                }
                ttk::mma_commit(bar_mma);
                w = ttk::mbar_wait(bar_mma, 0);
            }
            *sh_flag = w ? 1 : 0;
        }
        __syncthreads();
        if (*sh_flag == 0) {
            ok = false;
            break;
        }
        ttk::tc_fence_after();

        // ---- softmax on this thread's row
        uint32_t s0[32], s1[32];
        ttk::tmem_ld32(tS + lane_off + 0, s0);
        ttk::tmem_ld32(tS + lane_off + 32, s1);
        ttk::tmem_ld_wait32(s0);
        tie32(s1);
        const int lim = ctx - t * kTileKeys;  // keys at or past lim are outside the context
        float x[64];
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const float v = __uint_as_float(c < 32 ? s0[c] : s1[c - 32]) * g.scale_log2;
            x[c] = (c < lim) ? v : -CUDART_INF_F;
            mx = fmaxf(mx, x[c]);
        }
        if (j == 0) {
            m_run = mx;
        } else {
            const bool need = mx > m_run + kRescaleThreshold;
            if (__any_sync(0xffffffffu, need)) {
                const float alpha = need ? exp2f(m_run - mx) : 1.0f;
                if (need) {
                    m_run = mx;
                    l_run *= alpha;
                }
#pragma unroll
                for (int cc = 0; cc < D; cc += 32) {
                    uint32_t o[32];
                    ttk::tmem_ld32(tO + lane_off + cc, o);
                    ttk::tmem_ld_wait32(o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    ttk::tmem_st32(tO + lane_off + cc, o);
                }
                ttk::tmem_st_wait();
            }
        }
        float lsum = 0.f;
        uint8_t* prow = smem + L::kP + row_local * 128;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float p0 = exp2f(x[8 * c8 + 2 * e] - m_run);
                const float p1 = exp2f(x[8 * c8 + 2 * e + 1] - m_run);
                const __nv_bfloat162 pr = __floats2bfloat162_rn(p0, p1);
                lsum += __low2float(pr) + __high2float(pr);
                w4[e] = *reinterpret_cast<const uint32_t*>(&pr);
            }
            *reinterpret_cast<uint4*>(prow + ((c8 ^ (row_local & 7)) << 4)) =
                make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        l_run += lsum;
        if (lim < kTileKeys) {
            // Last tile of a context that ends inside it: the V rows past the end are
            // whatever the cache holds there (another sequence, an unused page slot).
            // P is 0 for them, but 0 * NaN would still poison O, so zero those rows.
            constexpr int kChunksPerRow = NP * 8;  // 16-byte chunks per V row
            uint8_t* vst = smem + L::kV + stage * L::kStage;
            for (int i = tid; i < (kTileKeys - lim) * kChunksPerRow; i += kSplitThreads) {
                const int key = lim + i / kChunksPerRow;
                const int ch = i % kChunksPerRow;
                *reinterpret_cast<uint4*>(vst + (ch >> 3) * L::kKVPart + key * 128 + ((ch & 7) << 4)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        ttk::fence_proxy_async_smem();
        ttk::tc_fence_before();
        __syncthreads();

        // ---- O += P V
        if (tid == 0) {
            ttk::tc_fence_after();
#pragma unroll
            for (int k = 0; k < kTileKeys / 16; ++k) {
                const uint64_t a = ttk::sdesc_sw128(sP + k * 32, 16, 1024);
                const uint64_t bd = ttk::sdesc_sw128(sV + stage * L::kStage + k * 2048, L::kKVPart, 1024);
                ttk::mma_bf16_ss(tO, a, bd, kIdescPV, (j > 0 || k > 0) ? 1u : 0u);
            }
            ttk::mma_commit(bar_mma);
            *sh_flag = ttk::mbar_wait(bar_mma, 1) ? 1 : 0;
        }
        __syncthreads();
        if (*sh_flag == 0) {
            ok = false;
            break;
        }
        ttk::tc_fence_after();
    }

    if (ok) {
        // tcgen05.ld is warp-collective: every lane loads, only rows in range store.
        float* acc = p.part_acc + pidx * D;
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
            uint32_t o[32];
            ttk::tmem_ld32(tO + lane_off + cc, o);
            ttk::tmem_ld_wait32(o);
            if (row_valid) {
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(acc + cc + e) =
                        make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                                    __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
            }
        }
        if (row_valid) {
            p.part_ml[2 * pidx + 0] = m_run;
            p.part_ml[2 * pidx + 1] = l_run;
        }
    } else {
        if (tid == 0) ttk::report_error(p.err, ttk::kErrTimeout);
        if (row_valid) {
            p.part_ml[2 * pidx + 0] = -CUDART_INF_F;
            p.part_ml[2 * pidx + 1] = 0.f;
        }
    }
    ttk::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ttk::tc_fence_after();
        ttk::tmem_dealloc(tmem, L::kTmemCols);
    }
}

// ---------------------------------------------------------------------------------
// Merge: partial states of the context splits + the S block keys -> out, lse.
// ---------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(512) attn_merge_kernel(const __grid_constant__ AttnMergeParams p) {
    constexpr int PER = D / 32;  // head dims per lane
    const AttnGeom& g = p.g;
    const int s = blockIdx.x, gkv = blockIdx.y, b = blockIdx.z;
    if (p.skip_if_zero != nullptr && __ldg(p.skip_if_zero + b) == 0) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int cap = g.page_size ? g.max_pages * g.page_size : g.max_ctx;
    int ctx = p.ctx_len ? __ldg(p.ctx_len + b) : g.max_ctx;
    if (ctx < 0 || ctx > cap) ctx = 0;  // reported by the split pass
    const int n_tiles = (ctx + kTileKeys - 1) / kTileKeys;
    const int n_valid = (n_tiles + g.tiles_per_split - 1) / g.tiles_per_split;

    for (int j = warp; j < g.G; j += nwarps) {
        const int h = gkv * g.G + j;
        const int r = s * g.G + j;
        // query row slice
        float q[PER];
        {
            const uint16_t* qp = p.q + (((size_t)b * g.S + s) * g.Hq + h) * D + lane * PER;
#pragma unroll
            for (int e = 0; e < PER; ++e) q[e] = ttk::bf16_bits_to_f32(qp[e]);
        }
        // block keys: lane k ends up holding the scaled logit of block key k
        float xk = -CUDART_INF_F;
        for (int k = 0; k < g.S; ++k) {
            const uint16_t* kp = p.k_blk + (((size_t)b * g.S + k) * g.Hkv + gkv) * D + lane * PER;
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < PER; ++e) d = fmaf(q[e], ttk::bf16_bits_to_f32(kp[e]), d);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (lane == k) xk = d * g.scale_log2;
        }
        // split states: lanes read (m_c, l_c) for c = lane, lane + 32, ...
        const size_t base = ((size_t)(b * g.Hkv + gkv) * g.n_splits) * (size_t)g.R + (size_t)r;
        float mloc = xk;
        for (int c = lane; c < n_valid; c += 32)
            mloc = fmaxf(mloc, __ldcg(p.part_ml + 2 * (base + (size_t)c * g.R)));
        float m = mloc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float acc[PER];
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = 0.f;
        float lloc = (lane < g.S) ? exp2f(xk - m) : 0.f;
        const float wk = lloc;
        for (int c0 = 0; c0 < n_valid; c0 += 32) {
            const int c = c0 + lane;
            float wc = 0.f;
            if (c < n_valid) {
                const size_t pi = base + (size_t)c * g.R;
                const float mc = __ldcg(p.part_ml + 2 * pi);
                if (mc != -CUDART_INF_F) {
                    wc = exp2f(mc - m);
                    lloc = fmaf(wc, __ldcg(p.part_ml + 2 * pi + 1), lloc);
                }
            }
            const int nc = min(32, n_valid - c0);
#pragma unroll 4
            for (int cc = 0; cc < nc; ++cc) {
                const float w = __shfl_sync(0xffffffffu, wc, cc);
                if (w != 0.f) {
                    const float* ap = p.part_acc + (base + (size_t)(c0 + cc) * g.R) * D + lane * PER;
                    if (PER == 4) {
                        const float4 a4 = __ldcg(reinterpret_cast<const float4*>(ap));
                        acc[0] = fmaf(w, a4.x, acc[0]);
                        acc[1] = fmaf(w, a4.y, acc[1]);
                        acc[2 % PER] = fmaf(w, a4.z, acc[2 % PER]);
                        acc[3 % PER] = fmaf(w, a4.w, acc[3 % PER]);
                    } else {
                        const float2 a2 = __ldcg(reinterpret_cast<const float2*>(ap));
                        acc[0] = fmaf(w, a2.x, acc[0]);
                        acc[1 % PER] = fmaf(w, a2.y, acc[1 % PER]);
                    }
                }
            }
        }
        float l = lloc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        for (int k = 0; k < g.S; ++k) {
            const float w = __shfl_sync(0xffffffffu, wk, k);
            const uint16_t* vp = p.v_blk + (((size_t)b * g.S + k) * g.Hkv + gkv) * D + lane * PER;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, ttk::bf16_bits_to_f32(vp[e]), acc[e]);
        }
        const float inv = 1.0f / l;
        uint16_t* op = p.out + (((size_t)b * g.S + s) * g.Hq + h) * D + lane * PER;
#pragma unroll
        for (int e = 0; e < PER; e += 2) {
            const __nv_bfloat162 pr = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
            *reinterpret_cast<uint32_t*>(op + e) = *reinterpret_cast<const uint32_t*>(&pr);
        }
        if (p.lse != nullptr && lane == 0)
            p.lse[((size_t)b * g.S + s) * g.Hq + h] = (m + log2f(l)) * 0.6931471805599453f;
    }
}

}  // namespace

bool attn_geometry(int B, int S, int Hq, int Hkv, int D, int max_ctx, int page_size,
                   int max_pages, int num_pages, float softmax_scale, int num_splits,
                   AttnGeom& g, const char** why) {
    *why = nullptr;
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || D < 1) { *why = "B, S, Hq, Hkv, D must be positive"; return false; }
    if (Hq % Hkv != 0) { *why = "Hq must be a multiple of Hkv"; return false; }
    g.B = B; g.S = S; g.Hq = Hq; g.Hkv = Hkv; g.G = Hq / Hkv; g.D = D;
    if (D != 64 && D != 128) { *why = "D must be 64 or 128"; return false; }
    if (S > 32) { *why = "S must be at most 32"; return false; }
    if (g.G > 128) { *why = "Hq/Hkv must be at most 128"; return false; }
    if (g.G * S > 512) { *why = "(Hq/Hkv)*S must be at most 512"; return false; }
    g.s_per_tile = (128 / g.G < S) ? 128 / g.G : S;
    g.rows_per_tile = g.s_per_tile * g.G;
    g.n_row_tiles = (S + g.s_per_tile - 1) / g.s_per_tile;
    g.R = g.G * S;
    g.page_size = page_size;
    g.max_pages = max_pages;
    g.num_pages = num_pages;
    if (page_size != 0) {
        if (page_size != 64) { *why = "page_size must be 0 or 64"; return false; }
        if (max_pages < 1 || num_pages < 1) { *why = "max_pages and num_pages must be positive"; return false; }
        if ((long long)max_pages * 64 > (1LL << 30)) { *why = "max_pages too large"; return false; }
        if ((long long)num_pages * 64 > (1LL << 31) - 64) { *why = "page pool too large"; return false; }
        g.max_ctx = max_pages * 64;
    } else {
        if (max_ctx < 0) { *why = "max_ctx must be >= 0"; return false; }
        if ((long long)B * max_ctx > (1LL << 31) - 64) { *why = "B*max_ctx too large"; return false; }
        g.max_ctx = max_ctx;
    }
    if (!(softmax_scale > 0.f) || !(softmax_scale < 1e30f)) { *why = "softmax_scale must be positive and finite"; return false; }
    g.scale_log2 = softmax_scale * kLog2e;
    const int n_tiles = (g.max_ctx + kTileKeys - 1) / kTileKeys;
    const long long items = (long long)B * Hkv * g.n_row_tiles;
    int tps;
    if (num_splits > 0) {
        tps = n_tiles > 0 ? (n_tiles + num_splits - 1) / num_splits : 1;
    } else {
        const long long target = 148LL * 2;
        long long want = (target + items - 1) / items;
        if (want < 1) want = 1;
        tps = (int)((n_tiles + want - 1) / want);
        if (tps > 64) tps = 64;
    }
    if (tps < 1) tps = 1;
    g.tiles_per_split = tps;
    g.n_splits = n_tiles > 0 ? (n_tiles + tps - 1) / tps : 1;
    if (g.n_splits > 65535) { *why = "too many context splits"; return false; }
    return true;
}

size_t attn_workspace_bytes(const AttnGeom& g) {
    const size_t rows = (size_t)g.B * g.Hkv * g.n_splits * g.R;
    size_t acc = rows * g.D * sizeof(float);
    acc = (acc + 255) & ~size_t(255);
    return acc + rows * 2 * sizeof(float) + 256;
}

cudaError_t attn_split_prepare(int D) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static unsigned long long done64 = 0, done128 = 0;  // one bit per device ordinal
    unsigned long long& done = (D == 128) ? done128 : done64;
    if (dev >= 0 && dev < 64 && ((done >> dev) & 1ull)) return cudaSuccess;
    if (D == 128)
        e = cudaFuncSetAttribute(attn_split_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SplitSmem<128>::kBytes);
    else
        e = cudaFuncSetAttribute(attn_split_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SplitSmem<64>::kBytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done |= (1ull << dev);
    return e;
}

cudaError_t launch_attn_split(const AttnSplitParams& p, const AttnMaps& maps, cudaStream_t stream) {
    const AttnGeom& g = p.g;
    dim3 grid(g.n_splits, g.Hkv * g.n_row_tiles, g.B);
    if (g.D == 128)
        attn_split_kernel<128><<<grid, kSplitThreads, SplitSmem<128>::kBytes, stream>>>(p, maps.q, maps.k, maps.v);
    else
        attn_split_kernel<64><<<grid, kSplitThreads, SplitSmem<64>::kBytes, stream>>>(p, maps.q, maps.k, maps.v);
    return cudaGetLastError();
}

cudaError_t launch_attn_merge(const AttnMergeParams& p, cudaStream_t stream) {
    const AttnGeom& g = p.g;
    dim3 grid(g.S, g.Hkv, g.B);
    const int warps = g.G < 16 ? g.G : 16;
    if (g.D == 128)
        attn_merge_kernel<128><<<grid, warps * 32, 0, stream>>>(p);
    else
        attn_merge_kernel<64><<<grid, warps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace tti
