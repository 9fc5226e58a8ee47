// LM head fused with confidence unmasking: the logits of the masked positions are
// formed on the tensor cores and reduced on the fly, so they never reach memory.
//
// "Nemotron-Labs-TwoTower" wiki, "Block-wise generation": every step predicts all
// masked positions of the block (the LM head over their hidden rows), then commits
// the confident ones.  logit[r][j] = sum_k h[r][k] * W[j][k] with W [V][H] (one row
// per token id), bf16 operands, fp32 accumulation.
//
// Three kernels, chained with programmatic dependent launch:
//  1. lmhead_gather_kernel: every CTA scans ids (B*S <= 4096) for the masked rows and
//     their compact order; its warps copy their rows' hidden vectors to the compact
//     matrix a_c, and CTA 0 publishes dest[] and the row count.
//  2. gemm_kernel<false>: one persistent CTA per SM.  A work item is (128-row tile of
//     a_c, vocabulary chunk); the chunks split the vocabulary in 64-id units so that
//     items = row tiles x chunks covers the CTAs once.  Per 256-id vocabulary tile:
//     warp 0 streams the A tile (128 rows x 64 of H) and four 64-row boxes of W per
//     64-wide slice of H into a four-stage ring (TMA, 128-byte swizzle; narrower
//     problems use tiles of one to three boxes, fewer rows of A when there are fewer
//     than 128, and up to 16 stages); warp 1 issues
//     tcgen05.mma 128 x 256 x 16 into one of two TMEM accumulators (256 columns each,
//     so the epilogue of one tile overlaps the products of the next); warps 2-5 (one
//     TMEM lane = one row per thread) read the accumulator and fold it into the row's
//     running (max, sum of 2^((x - max) * log2(e) / tau), lowest argmax), with the
//     mask id and ids past the chunk masked out.  Each item ends with one 16-byte
//     partial per row.
//  3. lmhead_finish_kernel: one CTA per sequence; a warp merges each masked row's
//     chunk partials, then warp 0 takes the sampler's commit/remask decision in place
//     (the same decision code as the unmask kernel).
// gemm_kernel<true> is the same GEMM with a bf16 store epilogue: the query/key/value
// projection of the adaLN output ("Architecture": the block's queries and its own
// keys/values are the denoiser's projections of its hidden states).
// Every wait on an mbarrier is bounded; one that runs out sets the error word, the
// roles drain what they issued, and TMEM is released.
#include <math_constants.h>

#include <mutex>

#include "tt_device.cuh"
#include "tt_internal.h"
#include "unmask_common.cuh"

namespace tti {
namespace {

using namespace um;

constexpr uint32_t kATile = 128 * 128;                  // 128 rows x 64 bf16
constexpr uint32_t kBBox = 64 * 128;                    // 64 vocabulary rows x 64 bf16
constexpr uint32_t kRingBytes = 4 * (kATile + 4 * kBBox);  // four stages of the widest tile
constexpr int kMaxStages = 16;
constexpr uint32_t kBarOff = kRingBytes;                // barriers after the ring
constexpr uint32_t kSlotOff = kBarOff + 512;            // TMEM address slot
constexpr uint32_t kSmemBytes = kBarOff + 1024 + 1024;  // + slack for 1024-B alignment
static_assert(8 * (2 * kMaxStages + 5) <= 512, "barriers fit before the TMEM slot");
constexpr int kGemmThreads = 192;                       // producer, MMA, 4 epilogue warps
constexpr int kGatherRows = 8;                          // rows copied per gather CTA (one per warp)

// Work split shared by the GEMM and the finish kernel.
struct Plan {
    int n_mt;      // 128-row tiles of the compact matrix
    int units;     // 64-id vocabulary units
    int n_chunks;  // vocabulary chunks per row tile
};
__device__ __forceinline__ Plan make_plan(int n_rows, int V, int n_ctas) {
    Plan pl;
    pl.n_mt = (n_rows + 127) / 128;
    pl.units = (V + 63) / 64;
    pl.n_chunks = pl.n_mt ? max(1, min(pl.units, n_ctas / pl.n_mt)) : 0;
    return pl;
}

// One persistent GEMM, two epilogues: the LM head's softmax reduction (per-row chunk
// partials) and the projection's bf16 store into up to three column segments.
struct GemmArgs {
    const int32_t* n_rows_dev;  // rows counted on the device, or null: n_rows
    int n_rows;
    int H, N;                   // reduction extent, output columns
    int n_ctas;
    UnmaskPartial* part;        // reduction: [rows][n_chunks]
    float temp_scale;
    int32_t mask_id;
    uint16_t* out[3];           // store: column segments [0, c0), [c0, c0 + c1), [.., N)
    int seg_cols[3];
    int* err;
};

__global__ void __launch_bounds__(256) lmhead_gather_kernel(LmHeadParams p) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    __shared__ int sdest[kLmHeadMaxRows];
    __shared__ int wsum[8];
    const int n = p.rows, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t* ids = p.um.ids;
    const int mask = p.um.mask_id;
    // thread t owns rows [t * per, (t + 1) * per): count, block-wide exclusive scan, write
    const int per = (n + 255) / 256;
    const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
    int cnt = 0;
    for (int i = i0; i < i1; ++i) cnt += (__ldcg(ids + i) == mask) ? 1 : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int base = 0, total = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        base += (w < warp) ? wsum[w] : 0;
        total += wsum[w];
    }
    int run = base + incl - cnt;
    for (int i = i0; i < i1; ++i) {
        const bool m = __ldcg(ids + i) == mask;
        sdest[i] = m ? run : -1;
        run += m ? 1 : 0;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int i = tid; i < n; i += 256) p.dest[i] = sdest[i];
        if (tid == 0) *p.n_rows = total;
    }
    const int row = blockIdx.x * kGatherRows + warp;
    if (warp < kGatherRows && row < n && sdest[row] >= 0) {
        // Eight 16-byte loads per lane in flight before any store (2688 bf16 = two rounds).
        const uint4* __restrict__ src = reinterpret_cast<const uint4*>(p.h + (size_t)row * p.H);
        uint4* __restrict__ dst = reinterpret_cast<uint4*>(p.a_c + (size_t)sdest[row] * p.H);
        const int n16 = p.H / 8;
        for (int c0 = lane; c0 < n16; c0 += 32 * 8) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c0 + 32 * u < n16) v[u] = __ldcg(src + c0 + 32 * u);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c0 + 32 * u < n16) dst[c0 + 32 * u] = v[u];
        }
    }
}

// All lanes of a warp agree on a bounded wait (tcgen05.ld below is warp-collective).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, ttk::mbar_wait(bar, parity));
}

template <bool kStore>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ LmHeadMaps maps, const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = ttk::smem_u32(smem);
    const uint32_t bar0 = sbase + kBarOff;
    auto full_bar = [&](uint32_t st) { return bar0 + 8u * st; };
    auto empty_bar = [&](uint32_t st) { return bar0 + 8u * (kMaxStages + st); };
    auto accf_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kMaxStages + a); };
    auto acce_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kMaxStages + 2 + a); };
    const uint32_t done_bar = bar0 + 8u * (2 * kMaxStages + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSlotOff);

    if (warp == 1) {
        ttk::tmem_alloc(ttk::smem_u32(tmem_slot), 512);
        ttk::tmem_relinquish();
    }
    if (tid == 0) {
        for (uint32_t st = 0; st < kMaxStages; ++st) {
            ttk::mbar_init(full_bar(st), 1);
            ttk::mbar_init(empty_bar(st), 1);
        }
        for (uint32_t a = 0; a < 2; ++a) {
            ttk::mbar_init(accf_bar(a), 1);
            ttk::mbar_init(acce_bar(a), 128);
        }
        ttk::mbar_init(done_bar, 1);
        ttk::fence_mbar_init();
        ttk::prefetch_tensormap(&maps.a);
        ttk::prefetch_tensormap(&maps.w);
    }
    ttk::tc_fence_before();
    __syncthreads();
    ttk::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    ttk::pdl_wait();  // the producer of A (gather or adaLN kernel) has completed
    ttk::pdl_trigger();
    const int n_rows = g.n_rows_dev ? __ldcg(g.n_rows_dev) : g.n_rows;
    const Plan pl = make_plan(n_rows, g.N, g.n_ctas);
    const int items = pl.n_mt * pl.n_chunks;
    const int nkb = (g.H + 63) / 64;
    // Vocabulary tiles are wbox 64-id units wide (the widest chunk needs no more).  A
    // stage holds the A box (maps.a_rows rows: below one 128-row tile only the rows
    // that exist) and wbox boxes of W; the ring holds as many stages as fit, up to 16,
    // so narrow problems keep more k-slices in flight.  The MMA reads 128 rows of A
    // from the stage; rows past a_rows read whatever follows (their accumulator rows
    // are never used), so the last stage keeps a whole tile of room below the ring's end.
    const int wbox = pl.n_chunks ? min(4, (pl.units + pl.n_chunks - 1) / pl.n_chunks) : 4;
    const uint32_t a_bytes = (uint32_t)maps.a_rows * 128u;
    // One k-slice: the A box then the W boxes.  Narrow slices are grouped kps to a
    // stage, so one barrier round trip (TMA completion, MMA commit, producer wake-up)
    // covers kps slices of products.
    const uint32_t slice_bytes = a_bytes + (uint32_t)wbox * kBBox;
    const int kps = slice_bytes <= 12u * 1024u ? 4 : slice_bytes <= 24u * 1024u ? 2 : 1;
    const uint32_t stage_bytes = (uint32_t)kps * slice_bytes;
    // the last stage's last slice needs a whole A tile of room (see above)
    const uint32_t tail = kATile + (uint32_t)(kps - 1) * slice_bytes;
    const uint32_t n_stages = min(min((uint32_t)kMaxStages, kRingBytes / stage_bytes),
                                  (kRingBytes - tail) / stage_bytes + 1u);
    const uint32_t idesc = ttk::idesc_bf16(128, 64 * wbox, false, false);
    bool ok = true;

    // item -> (row tile, chunk, first and end unit of the chunk)
    auto item_geom = [&](int item, int& mt, int& chunk, int& u0, int& u1) {
        mt = item % pl.n_mt;
        chunk = item / pl.n_mt;
        u0 = (int)((long long)chunk * pl.units / pl.n_chunks);
        u1 = (int)((long long)(chunk + 1) * pl.units / pl.n_chunks);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t kc = 0, st = 0, ph = 0;  // stages filled; ring slot and lap parity
            for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
                int mt, chunk, u0, u1;
                item_geom(item, mt, chunk, u0, u1);
                for (int ut = u0; ut < u1 && ok; ut += wbox) {
                    const int nbox = min(wbox, u1 - ut);
                    for (int kb = 0; kb < nkb; kb += kps, ++kc) {
                        if (kc >= n_stages && !ttk::mbar_wait(empty_bar(st), ph ^ 1u)) {
                            ok = false;
                            break;
                        }
                        if (kps == 1) {
                            const uint32_t sA = sbase + st * stage_bytes, sB = sA + a_bytes;
                            ttk::mbar_arrive_expect_tx(full_bar(st), a_bytes + (uint32_t)nbox * kBBox);
                            ttk::tma_load_2d(sA, &maps.a, kb * 64, mt * 128, full_bar(st));
                            for (int i = 0; i < nbox; ++i)
                                ttk::tma_load_2d(sB + (uint32_t)i * kBBox, &maps.w, kb * 64, (ut + i) * 64, full_bar(st));
                        } else {
                            const int ns = min(kps, nkb - kb);  // k-slices in this stage
                            ttk::mbar_arrive_expect_tx(full_bar(st), (uint32_t)ns * (a_bytes + (uint32_t)nbox * kBBox));
                            for (int s2 = 0; s2 < ns; ++s2) {
                                const uint32_t sA = sbase + st * stage_bytes + (uint32_t)s2 * slice_bytes;
                                const uint32_t sB = sA + a_bytes;
                                ttk::tma_load_2d(sA, &maps.a, (kb + s2) * 64, mt * 128, full_bar(st));
                                for (int i = 0; i < nbox; ++i)
                                    ttk::tma_load_2d(sB + (uint32_t)i * kBBox, &maps.w, (kb + s2) * 64, (ut + i) * 64,
                                                     full_bar(st));
                            }
                        }
                        if (++st == n_stages) {
                            st = 0;
                            ph ^= 1u;
                        }
                    }
                }
            }
            if (!ok) ttk::report_error(g.err, ttk::kErrTimeout);
            // Drain: the loads of the most recent stages have landed before exit.
            for (uint32_t j = (kc > n_stages) ? kc - n_stages : 0u; j < kc; ++j)
                ttk::mbar_wait(full_bar(j % n_stages), (j / n_stages) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, st = 0, ph = 0;  // ring slot and lap parity
            for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
                int mt, chunk, u0, u1;
                item_geom(item, mt, chunk, u0, u1);
                for (int ut = u0; ut < u1 && ok; ut += wbox, ++it) {
                    const uint32_t a = it & 1u;
                    if (it >= 2 && !ttk::mbar_wait(acce_bar(a), ((it >> 1) - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    ttk::tc_fence_after();
                    for (int kb = 0; kb < nkb; kb += kps) {
                        if (!ttk::mbar_wait(full_bar(st), ph)) {
                            ok = false;
                            break;
                        }
                        ttk::tc_fence_after();
                        if (kps == 1) {  // the issue loop of wide tiles stays as short as it can be
                            const uint32_t sA = sbase + st * stage_bytes, sB = sA + a_bytes;
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                ttk::mma_bf16_ss(tmem + a * 256u, ttk::sdesc_sw128(sA + 32u * k, 16, 1024),
                                                 ttk::sdesc_sw128(sB + 32u * k, 16, 1024), idesc,
                                                 (kb > 0 || k > 0) ? 1u : 0u);
                        } else {
                            const int ns = min(kps, nkb - kb);
                            for (int s2 = 0; s2 < ns; ++s2) {
                                const uint32_t sA = sbase + st * stage_bytes + (uint32_t)s2 * slice_bytes;
                                const uint32_t sB = sA + a_bytes;
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    ttk::mma_bf16_ss(tmem + a * 256u, ttk::sdesc_sw128(sA + 32u * k, 16, 1024),
                                                     ttk::sdesc_sw128(sB + 32u * k, 16, 1024), idesc,
                                                     (kb + s2 > 0 || k > 0) ? 1u : 0u);
                            }
                        }
                        ttk::mma_commit(empty_bar(st));  // this stage is no longer read
                        if (++st == n_stages) {
                            st = 0;
                            ph ^= 1u;
                        }
                    }
                    if (ok) ttk::mma_commit(accf_bar(a));
                }
            }
            if (!ok) ttk::report_error(g.err, ttk::kErrTimeout);
            // Everything issued has completed before shared memory and TMEM are released.
            ttk::mma_commit(done_bar);
            ttk::mbar_wait(done_bar, 0);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;  // warps 2, 3, 4, 5 -> TMEM lanes 64, 96, 0, 32
        const int lane_row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint32_t it = 0;
        for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
            int mt, chunk, u0, u1;
            item_geom(item, mt, chunk, u0, u1);
            const int vend = min(g.N, u1 * 64);
            const int row = mt * 128 + lane_row;
            Red acc{-CUDART_INF_F, 0.f, 0x7fffffff};
            for (int ut = u0; ut < u1; ut += wbox, ++it) {
                const uint32_t a = it & 1u;
                if (!warp_wait(accf_bar(a), (it >> 1) & 1u)) {
                    ok = false;
                    break;
                }
                ttk::tc_fence_after();
                const int v = ut * 64;
#pragma unroll 1
                for (int c = 0; c < 2 * wbox; ++c) {
                    uint32_t r[32];
                    ttk::tmem_ld32(tmem + lane_off + a * 256u + 32u * c, r);
                    ttk::tmem_ld_wait32(r);
                    const int col0 = v + 32 * c;
                    if constexpr (kStore) {
                        // 32 columns lie in one segment (segment widths are multiples of 64)
                        if (row < n_rows && col0 < vend) {
                            const int c01 = g.seg_cols[0] + g.seg_cols[1];
                            uint16_t* base = (col0 < g.seg_cols[0]) ? g.out[0] : (col0 < c01) ? g.out[1] : g.out[2];
                            const int width = (col0 < g.seg_cols[0]) ? g.seg_cols[0] : (col0 < c01) ? g.seg_cols[1] : g.seg_cols[2];
                            const int c_in = col0 - ((col0 < g.seg_cols[0]) ? 0 : (col0 < c01) ? g.seg_cols[0] : c01);
                            uint4* dst = reinterpret_cast<uint4*>(base + (size_t)row * width + c_in);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                uint32_t w[4];
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const __nv_bfloat162 pr = __floats2bfloat162_rn(
                                        __uint_as_float(r[8 * q4 + 2 * u]), __uint_as_float(r[8 * q4 + 2 * u + 1]));
                                    w[u] = *reinterpret_cast<const uint32_t*>(&pr);
                                }
                                dst[q4] = make_uint4(w[0], w[1], w[2], w[3]);
                            }
                        }
                    } else {
                        float x[32];
                        int id[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int col = col0 + e;
                            id[e] = col;
                            x[e] = (col < vend && col != g.mask_id) ? __uint_as_float(r[e]) : -CUDART_INF_F;
                        }
                        fold<32>(acc, x, id, g.temp_scale);
                    }
                }
                ttk::tc_fence_before();
                ttk::mbar_arrive(acce_bar(a));
            }
            if (!ok) break;
            if constexpr (!kStore) {
                if (row < n_rows)
                    __stcg(reinterpret_cast<float4*>(g.part + (size_t)row * pl.n_chunks + chunk), as_f4(acc));
            }
        }
        if (!ok) ttk::report_error(g.err, ttk::kErrTimeout);
    }
    ttk::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ttk::tc_fence_after();
        ttk::tmem_dealloc(tmem, 512);
    }
}

// One CTA per sequence: warp w merges rows w, w + 8, ... (lanes stride over the row's
// chunk partials, so all its loads are in flight together), then warp 0 decides.
constexpr int kFinishThreads = 256;
__global__ void __launch_bounds__(kFinishThreads) lmhead_finish_kernel(LmHeadParams p) {
    ttk::pdl_wait();  // the GEMM's partials (and, through it, the gather's dest[])
    ttk::pdl_trigger();
    const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const UnmaskParams& u = p.um;
    const Plan pl = make_plan(__ldcg(p.n_rows), p.V, p.n_ctas);
    for (int s = warp; s < u.S; s += kFinishThreads / 32) {
        const int row = b * u.S + s;
        const int cr = __ldcg(p.dest + row);
        if (cr < 0) continue;  // warp-uniform
        const float4* pp = reinterpret_cast<const float4*>(p.part + (size_t)cr * pl.n_chunks);
        float4 v[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const int c = lane + 32 * i;
            v[i] = (c < pl.n_chunks) ? __ldcg(pp + c) : make_float4(-CUDART_INF_F, 0.f, __int_as_float(0x7fffffff), 0.f);
        }
        Red r = from_f4(v[0]);
#pragma unroll
        for (int i = 1; i < 5; ++i) r = combine(r, from_f4(v[i]), u.temp_scale);
        for (int c = lane + 160; c < pl.n_chunks; c += 32) r = combine(r, from_f4(__ldcg(pp + c)), u.temp_scale);
        r = warp_combine(r, u.temp_scale);
        if (lane == 0) __stcg(reinterpret_cast<float4*>(u.row_res) + row, as_f4(r));
    }
    __syncthreads();  // the row results are visible to warp 0
    if (warp == 0) decide(u, b);
}

std::mutex g_attr_mu;
unsigned long long g_attr_done = 0;  // one bit per device ordinal

cudaError_t gemm_prepare() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (dev >= 0 && dev < 64 && ((g_attr_done >> dev) & 1ull)) return cudaSuccess;
    e = cudaFuncSetAttribute(gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) g_attr_done |= (1ull << dev);
    return e;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

// The compact matrix has whole 128-row tiles, so every TMA box of it is in bounds.
size_t lmhead_a_rows(int rows) { return ((size_t)rows + 127) / 128 * 128; }

size_t lmhead_workspace_bytes(int B, int S, int H, int n_ctas) {
    const size_t rows = (size_t)B * S;
    return align256(lmhead_a_rows((int)rows) * H * 2)        // a_c
           + align256(rows * 4)                              // dest
           + 256                                             // n_rows
           + align256(rows * (size_t)n_ctas * sizeof(UnmaskPartial))  // chunk partials
           + align256(rows * sizeof(UnmaskPartial))          // row results
           + align256((rows + B + 1) * sizeof(unsigned int));  // decision tickets
}

void lmhead_layout(void* ws, LmHeadParams& p) {
    const size_t rows = (size_t)p.rows;
    char* w = static_cast<char*>(ws);
    p.a_c = reinterpret_cast<uint16_t*>(w);
    w += align256(lmhead_a_rows(p.rows) * p.H * 2);
    p.dest = reinterpret_cast<int32_t*>(w);
    w += align256(rows * 4);
    p.n_rows = reinterpret_cast<int32_t*>(w);
    w += 256;
    p.part = reinterpret_cast<UnmaskPartial*>(w);
    w += align256(rows * (size_t)p.n_ctas * sizeof(UnmaskPartial));
    p.um.row_res = reinterpret_cast<UnmaskPartial*>(w);
    w += align256(rows * sizeof(UnmaskPartial));
    p.um.ticket = reinterpret_cast<unsigned int*>(w);
    p.um.ticket_words = (int)rows + p.um.B;
    p.um.part = p.part;
}

cudaError_t lmhead_prepare() { return gemm_prepare(); }

cudaError_t launch_lmhead(const LmHeadParams& p, const LmHeadMaps& maps, cudaStream_t stream) {
    cudaError_t e = gemm_prepare();
    if (e != cudaSuccess) return e;
    const int n_gather = (p.rows + kGatherRows - 1) / kGatherRows;
    e = launch_pdl(lmhead_gather_kernel, dim3(n_gather), dim3(256), 0, stream, p);
    if (e != cudaSuccess) return e;
    GemmArgs g{};
    g.n_rows_dev = p.n_rows;
    g.n_rows = 0;
    g.H = p.H;
    g.N = p.V;
    g.n_ctas = p.n_ctas;
    g.part = p.part;
    g.temp_scale = p.um.temp_scale;
    g.mask_id = p.um.mask_id;
    g.err = p.um.err;
    e = launch_pdl(gemm_kernel<false>, dim3(p.n_ctas), dim3(kGemmThreads), (size_t)kSmemBytes, stream, maps, g);
    if (e != cudaSuccess) return e;
    return launch_pdl(lmhead_finish_kernel, dim3(p.um.B), dim3(kFinishThreads), 0, stream, p);
}

cudaError_t launch_qkv(const QkvParams& p, const LmHeadMaps& maps, cudaStream_t stream) {
    cudaError_t e = gemm_prepare();
    if (e != cudaSuccess) return e;
    GemmArgs g{};
    g.n_rows_dev = nullptr;
    g.n_rows = p.rows;
    g.H = p.H;
    g.N = (p.Hq + 2 * p.Hkv) * p.D;
    g.n_ctas = p.n_ctas;
    g.mask_id = -1;
    g.out[0] = p.q;
    g.out[1] = p.k;
    g.out[2] = p.v;
    g.seg_cols[0] = p.Hq * p.D;
    g.seg_cols[1] = p.Hkv * p.D;
    g.seg_cols[2] = p.Hkv * p.D;
    g.err = p.err;
    return launch_pdl(gemm_kernel<true>, dim3(p.n_ctas), dim3(kGemmThreads), (size_t)kSmemBytes, stream, maps, g);
}

}  // namespace tti
