// Denoise attention: split-KV pass over the context cache on tcgen05, then (when a
// row's context is split) a pass that combines the partial states.
//
// "Nemotron-Labs-TwoTower" wiki, "Architecture": block queries attend over the
// context tower's layer-i KV cache followed by the denoiser's own layer-i keys and
// values for the block, with bidirectional attention inside the block.
//
// Split pass, one CTA per (context split, row group, kv head, sequence):
//   * the rows are the packed (block position s, query head j of the GQA group)
//     pairs, row = s*G + j.  One CTA serves up to 256 of them as one or two 128-row
//     MMA tiles, so every K/V tile it loads feeds G*S query rows and QK^T / PV are
//     dense contractions (M = 128, N = 128 keys, K = D for QK^T; N = D, K = 128 for PV).
//     A call of only a few key tiles per SM in all is latency-bound and takes one
//     128-row tile per CTA instead (twice the CTAs, half the work per round);
//   * split 0 also takes the block's own S keys, as one extra (masked) key tile in
//     front of its context tiles, so the block keys run on the tensor cores too;
//   * warp 0 streams 128-token K/V tiles (two 64-row TMA boxes each, so a tile may
//     span two pages of a paged cache) into a shared-memory ring with 128-byte
//     swizzle; warp 1 issues every tcgen05.mma; four softmax warpgroups own the rows:
//     warpgroup (i, h) takes tile i's 128 rows (one per thread / TMEM lane) and keys
//     64h .. 64h+63 of every 128-key tile.  The two halves of a row agree on its max
//     through shared memory and a named barrier;
//   * Q sits in shared memory for the whole CTA; the scores S go to tensor memory
//     (TMEM); the softmax turns them into P = exp2(S*scale*log2e - m) (bf16) written
//     back over the front of each half's S columns, which is the TMEM A operand of
//     PV; O accumulates in
//     TMEM.  N = 128 keys per QK^T instruction keeps the tensor core near its peak
//     rate (64-key products run at little more than half of it);
//   * the two row tiles ping-pong: the MMA warp issues QK(0,j) QK(1,j) | PV(0,j)
//     QK(0,j+1) | PV(1,j) QK(1,j+1) | ..., so one tile's softmax overlaps the other's
//     matrix products;
//   * the running max is raised (and O rescaled in TMEM) only when it grows by more
//     than 2^8, so most tiles need no correction;
//   * a CTA whose row group has one non-empty split writes the normalised output
//     (bf16) and the lse itself; otherwise each row's partial state (m, l, O) goes to
//     the workspace and the combine pass (one warp per output row) merges them;
//   * on ragged paged batches of more than one wave a one-CTA prep kernel picks the
//     call's split length from the active sequences' lengths and sorts the work units
//     longest first; the split kernel's 1-D grid takes them in that order.
//
// Every wait is bounded: a wait that runs out sets the device error word, the CTA
// drains what it issued and returns.
#include <math_constants.h>

#include "tt_device.cuh"
#include "tt_internal.h"

namespace tti {
namespace {

constexpr int kTileKeys = 128;  // keys per pipeline round (two 64-token pages)
constexpr int kSub = 64;        // keys per TMA box (one page of a paged cache)
constexpr int kThreads = 640;   // warp 0 TMA, warp 1 MMA, warps 2-3 spare, 4-19 softmax
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Cfg {
    static constexpr int NP = D / 64;                      // 128-byte column parts of a row
    static constexpr uint32_t kPart = kTileKeys * 128;     // 128 rows x 128 B (one part of a tile)
    static constexpr uint32_t kTile = NP * kPart;          // one K (or V) tile
    static constexpr uint32_t kStage = 2 * kTile;          // K then V
    static constexpr int kStages = (D == 128) ? 2 : 4;     // K/V ring depth (128 KiB)
    static constexpr uint32_t kQPart = 128 * 128;          // 128 query rows x 128 B
    static constexpr uint32_t kQTile = NP * kQPart;        // one 128-row Q tile
    static constexpr uint32_t kRing = 2 * kQTile;          // Q tiles first, then the ring
    static constexpr uint32_t kXchg = kRing + kStages * kStage;  // float [2 tiles][2 halves][128]
    static constexpr uint32_t kBar = kXchg + 2 * 2 * 128 * 4;
    // mbarriers: k_full[st], v_full[st], k_empty[st], v_empty[st], s_full[2], p_full[2],
    // o_full, q_ready; then the TMEM slot.  K and V of a stage are tracked apart: K is
    // free again once both QK^T products have read it, a round before V.
    static constexpr int kNumBars = 4 * kStages + 6;
    static constexpr uint32_t kSlot = kBar + 8 * kNumBars;
    static constexpr uint32_t kEnd = kSlot + 16;
    static constexpr uint32_t kBytes = kEnd + 1024;        // alignment slack
    // TMEM columns (512 allocated): S_i at 128 i (P_i, bf16, over its first 64);
    // O_i at 256 + D i.
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColO = 256;
    // Epilogue staging: one half row (D/2 floats) per softmax thread, padded so the
    // 16-byte stores of consecutive rows fall in different banks.
    static constexpr uint32_t kHalfRow = D * 2 + 16;
    static_assert(kColO + 2 * D <= 512, "TMEM budget");
    static_assert(kBytes <= 227 * 1024, "shared memory budget");
    static_assert(512 * kHalfRow <= kXchg, "epilogue staging fits in the Q tiles + ring");
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

__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Combine inside the split pass (fused): every non-empty split CTA of a row group
// stores its partial state with plain stores, counts itself in on the group's ticket
// (release), waits until all nv splits have (acquire, bounded), and then merges its
// share of the group's rows, one softmax warp per row with every split's state in
// flight.  The launch is cooperative (all CTAs resident), so no CTA waits for one that
// cannot start.  The last CTA to finish resets the group's two counters.
template <int D>
__device__ __forceinline__ void fused_combine(const AttnSplitParams& p, uint32_t tO, int half, bool row_valid, int r_glob,
                                           int b, int gkv, int rg, int split, int nv, int n_mt, bool ok, float m_run,
                                           float l, int q, int lane_row, int tid, volatile int* s_go) {
    constexpr int PER = D / 32;
    const AttnGeom& g = p.g;
    const int n_thr = 256 * n_mt;  // the softmax threads of this CTA
    ttk::tc_fence_after();
    const size_t pi = ((size_t)(b * g.Hkv + gkv) * g.n_splits + split) * (size_t)g.R + r_glob;
#pragma unroll
    for (int cc = 0; cc < D / 2; cc += 32) {
        uint32_t o[32];
        ttk::tmem_ld32(tO + half * (D / 2) + cc, o);  // warp-collective: every lane loads
        ttk::tmem_ld_wait32(o);
        if (row_valid) {
            float4* dst = reinterpret_cast<float4*>(p.part_acc + pi * D + half * (D / 2) + cc);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                __stcg(dst + e, make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                            __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3])));
        }
    }
    if (row_valid && half == 0) {
        p.part_ml[2 * pi + 0] = ok ? m_run : -CUDART_INF_F;
        p.part_ml[2 * pi + 1] = ok ? l : 0.f;
    }
    __threadfence();
    named_sync(4, n_thr);  // this CTA's partial state is written
    const int rgi = (b * g.Hkv + gkv) * g.n_rg + rg;
    unsigned* arrive = p.ticket + rgi;
    unsigned* done = p.ticket + g.B * g.Hkv * g.n_rg + rgi;
    if (q == 0 && lane_row == 0) {
        unsigned v;
        asm volatile("atom.add.release.gpu.global.u32 %0, [%1], 1;" : "=r"(v) : "l"(arrive) : "memory");
        int go = 1;
        const uint64_t t0 = ttk::globaltimer();
        while (true) {
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(arrive) : "memory");
            if (v >= (unsigned)nv) break;
            if (ttk::globaltimer() - t0 > ttk::kWaitLimitNs) {
                go = 0;
                ttk::report_error(p.err, ttk::kErrTimeout);
                break;
            }
            __nanosleep(64);
        }
        *s_go = go;
    }
    named_sync(4, n_thr);
    if (*s_go != 0) {
        // the group's rows, split evenly over its nv CTAs; a warp per row
        const int lane = tid & 31;
        const int w = (tid >> 5) - 4, n_w = n_thr / 32;
        const int rg0 = rg * g.rows_per_cta;
        const int rows = min(g.rows_per_cta, g.R - rg0);
        const int r0 = (int)((long long)split * rows / nv), r1 = (int)((long long)(split + 1) * rows / nv);
        const size_t base = (size_t)(b * g.Hkv + gkv) * g.n_splits * (size_t)g.R;
        for (int r = r0 + w; r < r1; r += n_w) {
            const int row = rg0 + r;
            float m = -CUDART_INF_F, lsum = 0.f, acc[PER];
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] = 0.f;
            for (int c0 = 0; c0 < nv; c0 += 8) {
                const int nc = min(8, nv - c0);
                float mc[8], lc[8], a[8][PER];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const size_t pc = base + (size_t)(c0 + min(u, nc - 1)) * g.R + row;
                    const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + pc);
                    mc[u] = ml.x;
                    lc[u] = ml.y;
                    const float* ap = p.part_acc + pc * D + lane * PER;
                    if (PER == 4) {
                        const float4 v4 = __ldcg(reinterpret_cast<const float4*>(ap));
                        a[u][0] = v4.x; a[u][1 % PER] = v4.y; a[u][2 % PER] = v4.z; a[u][3 % PER] = v4.w;
                    } else {
                        const float2 v2 = __ldcg(reinterpret_cast<const float2*>(ap));
                        a[u][0] = v2.x; a[u][1 % PER] = v2.y;
                    }
                }
                float mn = m;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (u < nc) mn = fmaxf(mn, mc[u]);
                if (mn == -CUDART_INF_F) continue;
                if (m != -CUDART_INF_F && mn != m) {
                    const float rsc = exp2f(m - mn);
                    lsum *= rsc;
#pragma unroll
                    for (int e = 0; e < PER; ++e) acc[e] *= rsc;
                }
                m = mn;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (u >= nc || mc[u] == -CUDART_INF_F) continue;
                    const float wu = exp2f(mc[u] - m);
                    lsum = fmaf(wu, lc[u], lsum);
#pragma unroll
                    for (int e = 0; e < PER; ++e) acc[e] = fmaf(wu, a[u][e], acc[e]);
                }
            }
            const float inv = 1.0f / lsum;
            const int s = row / g.G, j = row % g.G;
            const size_t orow = ((size_t)b * g.S + s) * g.Hq + (size_t)gkv * g.G + j;
            uint16_t* op = p.out + orow * D + lane * PER;
#pragma unroll
            for (int e = 0; e < PER; e += 2) {
                const __nv_bfloat162 pr = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
                *reinterpret_cast<uint32_t*>(op + e) = *reinterpret_cast<const uint32_t*>(&pr);
            }
            if (p.lse != nullptr && lane == 0) p.lse[orow] = (m + log2f(lsum)) * kLn2;
        }
    }
    named_sync(4, n_thr);  // this CTA's merge reads are done
    if (q == 0 && lane_row == 0) {
        // every CTA of the group is past its wait once all have counted in here
        const unsigned old = atomicAdd(done, 1u);
        if (old == (unsigned)nv - 1u) {
            *arrive = 0u;
            *done = 0u;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_split_kernel(const __grid_constant__ AttnSplitParams p,
                      const __grid_constant__ AttnMaps maps) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    using C = Cfg<D>;
    constexpr int NP = C::NP;
    constexpr int NS = C::kStages;
    constexpr uint32_t kIdescQK = ttk::idesc_bf16(128, kTileKeys, false, false);
    constexpr uint32_t kIdescPV = ttk::idesc_bf16(128, D, false, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kSlot);
    float* xchg = reinterpret_cast<float*>(smem + C::kXchg);  // [tile][half][row]

    const AttnGeom& g = p.g;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    // Work unit u = item + n_items * split, item = rg + n_rg * (kv head + Hkv * sequence).
    // Grid: x = item, y = split, so splits vary slowest; on a ragged batch (lpt) a 1-D
    // grid takes the units longest first from the order the prep kernel sorted, and the
    // CTAs past the non-empty units exit.
    const int n_items = g.B * g.Hkv * g.n_rg;
    long long unit = (long long)blockIdx.y * n_items + blockIdx.x;
    int tps = g.tiles_per_split;
    if (p.order != nullptr) {
        const long long n_units = (long long)n_items * g.n_splits;
        if ((long long)blockIdx.x >= __ldg(p.order + n_units)) return;
        unit = __ldg(p.order + blockIdx.x);
        tps = __ldg(p.order + n_units + 1);  // this call's split length
    }
    const int item = (int)(unit % n_items);
    const int rg = item % g.n_rg;
    const int gkv = (item / g.n_rg) % g.Hkv;
    const int b = item / (g.n_rg * g.Hkv);
    const int split = (int)(unit / n_items);

    if (p.skip_if_zero != nullptr && __ldg(p.skip_if_zero + b) == 0) return;
    const int cap = g.page_size ? g.max_pages * g.page_size : g.max_ctx;
    const int ctx = p.ctx_len ? __ldg(p.ctx_len + b) : g.max_ctx;
    if (ctx < 0 || ctx > cap) {
        if (tid == 0 && split == 0 && rg == 0) ttk::report_error(p.err, ttk::kErrDevice);
        return;
    }
    // Tiles of this CTA: split 0 starts with the block's own keys, then context tiles
    // t0 .. t1-1.
    const int n_tiles = (ctx + kTileKeys - 1) / kTileKeys;
    const int t0 = split * tps;
    const int t1 = min(n_tiles, t0 + tps);
    const int nblk = (split == 0) ? 1 : 0;
    const int nt = nblk + max(0, t1 - t0);
    if (nt == 0) return;  // this split is empty; the combine pass does not read it
    const int n_mt = g.n_mt;
    // Direct: this CTA sees every key of its rows (its row group has one non-empty
    // split) and writes the normalised output itself; the combine pass skips the rows.
    const int nv = max(1, (n_tiles + tps - 1) / tps);
    const bool direct = g.n_splits == 1 || nv == 1;

    if (g.page_size && t1 > t0) {
        // Every page this split reads must exist; pages past the context end are not read.
        const int pg0 = t0 * 2;
        const int pg1 = min(t1 * 2, (ctx + kSub - 1) / kSub);
        int bad = 0;
        for (int t = pg0 + tid; t < pg1; t += kThreads) {
            const int pg = __ldg(p.page_table + (size_t)b * g.max_pages + t);
            bad |= (pg < 0 || pg >= g.num_pages) ? 1 : 0;
        }
        if (__syncthreads_or(bad)) {
            // Leave an empty partial state for every row so the combine skips this
            // split (a single-split call has no partials: its output is left unwritten).
            if (tid == 0) ttk::report_error(p.err, ttk::kErrDevice);
            if (!direct) {
                for (int r = tid; r < g.rows_per_cta; r += kThreads) {
                    const int rglob = rg * g.rows_per_cta + r;
                    if (rglob < g.R) {
                        const size_t pi = ((size_t)(b * g.Hkv + gkv) * g.n_splits + split) * (size_t)g.R + rglob;
                        p.part_ml[2 * pi + 0] = -CUDART_INF_F;
                        p.part_ml[2 * pi + 1] = 0.f;
                    }
                }
            }
            return;
        }
    }

    const uint32_t sQ = ttk::smem_u32(smem);
    const uint32_t sRing = ttk::smem_u32(smem + C::kRing);
    const uint32_t bar0 = ttk::smem_u32(smem + C::kBar);
    auto kfull_bar = [&](int st) { return bar0 + 8u * (uint32_t)st; };
    auto vfull_bar = [&](int st) { return bar0 + 8u * (uint32_t)(NS + st); };
    auto kempty_bar = [&](int st) { return bar0 + 8u * (uint32_t)(2 * NS + st); };
    auto vempty_bar = [&](int st) { return bar0 + 8u * (uint32_t)(3 * NS + st); };
    auto sfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(4 * NS + i); };
    auto pfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(4 * NS + 2 + i); };
    const uint32_t ofull_bar = bar0 + 8u * (uint32_t)(4 * NS + 4);
    const uint32_t qready_bar = bar0 + 8u * (uint32_t)(4 * NS + 5);

    if (warp == 1) {
        ttk::tmem_alloc(ttk::smem_u32(tmem_slot), 512);
        ttk::tmem_relinquish();
    }
    if (tid == 0) {
        for (int st = 0; st < NS; ++st) {
            ttk::mbar_init(kfull_bar(st), 1);
            ttk::mbar_init(vfull_bar(st), 1);
            ttk::mbar_init(kempty_bar(st), 1);
            ttk::mbar_init(vempty_bar(st), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ttk::mbar_init(sfull_bar(i), 1);
            ttk::mbar_init(pfull_bar(i), 256);
        }
        ttk::mbar_init(ofull_bar, 1);
        ttk::mbar_init(qready_bar, 128 * n_mt * NP);
        ttk::fence_mbar_init();
    }
    ttk::tc_fence_before();
    __syncthreads();
    ttk::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int q = warp / 4 - 1;            // softmax warpgroup 0..3, or -1 for warps 0-3
    const int mt = q >> 1;                 // its 128-row tile
    const int half = q & 1;                // its 64 keys of every 128-key tile
    const int lane_row = tid & 127;        // TMEM lane (tile row) of this softmax thread
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int r_local = mt * 128 + lane_row;               // row within this CTA
    const int r_glob = rg * g.rows_per_cta + r_local;      // packed row of (b, gkv)
    const bool in_tile = q >= 0 && mt < n_mt;
    const bool row_valid = in_tile && r_local < g.rows_per_cta && r_glob < g.R;

    bool ok = true;
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if ((tid & 31) == 0) {
            ttk::prefetch_tensormap(&maps.k);
            ttk::prefetch_tensormap(&maps.v);
            if (nblk) {
                ttk::prefetch_tensormap(&maps.kb);
                ttk::prefetch_tensormap(&maps.vb);
            }
            int issued[2] = {0, 0};  // K and V tiles whose loads were issued
            for (int j = 0; j < nt && ok; ++j) {
                const int st = j % NS;
                const uint32_t par = (uint32_t)(((j / NS) - 1) & 1);
                const uint32_t dK = sRing + (uint32_t)st * C::kStage;
                const bool blk = j < nblk;
                const int t = t0 + j - nblk;
                // First cache row of each 64-row half.  A second half past the end (the
                // block's S <= 32 keys, or the context end) re-reads the first half's
                // rows: they are masked out, every box stays in range, and no page past
                // the sequence is looked up.
                int row0[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (blk) {
                        row0[h] = b * g.S;
                    } else {
                        const int hh = (t * kTileKeys + h * kSub < ctx) ? h : 0;
                        row0[h] = g.page_size ? __ldg(p.page_table + (size_t)b * g.max_pages + 2 * t + hh) * kSub
                                              : b * g.max_ctx + t * kTileKeys + hh * kSub;
                    }
                }
#pragma unroll
                for (int kv = 0; kv < 2; ++kv) {  // K, then V
                    if (j >= NS && !ttk::mbar_wait(kv ? vempty_bar(st) : kempty_bar(st), par)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = kv ? vfull_bar(st) : kfull_bar(st);
                    const CUtensorMap* map = kv ? (blk ? &maps.vb : &maps.v) : (blk ? &maps.kb : &maps.k);
                    ttk::mbar_arrive_expect_tx(fb, C::kTile);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int part = 0; part < NP; ++part)
                            ttk::tma_load_3d(dK + kv * C::kTile + part * C::kPart + h * (kSub * 128), map,
                                             part * 64, gkv, row0[h], fb);
                    issued[kv] = j + 1;
                }
            }
            if (!ok) ttk::report_error(p.err, ttk::kErrTimeout);
            // Drain: the most recent loads of every stage must have landed before exit.
#pragma unroll
            for (int kv = 0; kv < 2; ++kv)
                for (int st = 0; st < NS && st < issued[kv]; ++st) {
                    const int jl = st + ((issued[kv] - 1 - st) / NS) * NS;
                    ttk::mbar_wait(kv ? vfull_bar(st) : kfull_bar(st), (uint32_t)((jl / NS) & 1));
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if ((tid & 31) == 0) {
            auto qk = [&](int i, int j) {
                const uint32_t sK = sRing + (uint32_t)(j % NS) * C::kStage;
                const uint32_t sQi = sQ + (uint32_t)i * C::kQTile;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t koff = (uint32_t)(k >> 2) * C::kPart + (k & 3) * 32;
                    const uint64_t ad = ttk::sdesc_sw128(sQi + (uint32_t)(k >> 2) * C::kQPart + (k & 3) * 32, 16, 1024);
                    const uint64_t bd = ttk::sdesc_sw128(sK + koff, 16, 1024);
                    ttk::mma_bf16_ss(tmem + C::kColS + 128 * i, ad, bd, kIdescQK, k > 0 ? 1u : 0u);
                }
                ttk::mma_commit(sfull_bar(i));
            };
            auto pv = [&](int i, int j) {
                const uint32_t sV = sRing + (uint32_t)(j % NS) * C::kStage + C::kTile;
#pragma unroll
                for (int k = 0; k < kTileKeys / 16; ++k) {
                    const uint64_t bd = ttk::sdesc_sw128(sV + k * 2048, C::kPart, 1024);
                    // keys 16k .. 16k+15: P of key half k/4 sits over the front of that
                    // half's own 64 S columns
                    const uint32_t pcol = C::kColS + 128 * i + 64 * (k >> 2) + 8 * (k & 3);
                    ttk::mma_bf16_ts(tmem + C::kColO + i * D, tmem + pcol, bd, kIdescPV,
                                     (j > 0 || k > 0) ? 1u : 0u);
                }
            };
            auto wait_k = [&](int j) { return ttk::mbar_wait(kfull_bar(j % NS), (uint32_t)((j / NS) & 1)); };
            auto wait_v = [&](int j) { return ttk::mbar_wait(vfull_bar(j % NS), (uint32_t)((j / NS) & 1)); };
            ok = ttk::mbar_wait(qready_bar, 0) && wait_k(0);
            if (ok) {
                ttk::tc_fence_after();
                qk(0, 0);
                if (n_mt == 2) qk(1, 0);
                ttk::mma_commit(kempty_bar(0));  // K of tile 0 is no longer read
            }
            for (int j = 0; j < nt && ok; ++j) {
                const uint32_t par = (uint32_t)(j & 1);
                if (!(ok = ttk::mbar_wait(pfull_bar(0), par) && wait_v(j))) break;
                ttk::tc_fence_after();
                pv(0, j);
                const bool next = j + 1 < nt;
                if (next) {
                    if (!(ok = wait_k(j + 1))) break;
                    ttk::tc_fence_after();
                    qk(0, j + 1);
                    if (n_mt == 1) ttk::mma_commit(kempty_bar((j + 1) % NS));
                }
                if (n_mt == 2) {
                    if (!(ok = ttk::mbar_wait(pfull_bar(1), par))) break;
                    ttk::tc_fence_after();
                    pv(1, j);
                }
                ttk::mma_commit(vempty_bar(j % NS));  // V of tile j is no longer read
                if (next && n_mt == 2) {
                    qk(1, j + 1);
                    ttk::mma_commit(kempty_bar((j + 1) % NS));
                }
            }
            if (!ok) ttk::report_error(p.err, ttk::kErrTimeout);
            // Completion of everything issued: the epilogue waits for it, and so does
            // this lane before the TMEM release below (also after a timeout).
            ttk::mma_commit(ofull_bar);
            ttk::mbar_wait(ofull_bar, 0);
        }
    } else if (in_tile) {
        // ---- this row's Q into shared memory (canonical K-major, 128-B swizzle)
        // Half h loads 128-byte part h of the row (D = 128: both halves, one part
        // each, so the whole row arrives in one round trip; D = 64: half 0 alone).
        if (half < NP) {
            const int s = r_glob / g.G, j = r_glob % g.G;
            const uint4* qp = reinterpret_cast<const uint4*>(
                p.q + (((size_t)b * g.S + s) * g.Hq + (size_t)gkv * g.G + j) * D) + half * 8;
            uint8_t* qrow = smem + (size_t)mt * C::kQTile + (size_t)half * C::kQPart + (size_t)lane_row * 128;
            uint4 qv[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) qv[c] = row_valid ? __ldg(qp + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(qrow + ((c ^ (lane_row & 7)) << 4)) = qv[c];
            ttk::fence_proxy_async_smem();
            ttk::mbar_arrive(qready_bar);
        }
        // ------------------------------------------------- softmax: tile mt, keys half
        const uint32_t tS = tmem + lane_off + C::kColS + 128 * mt;
        const uint32_t tO = tmem + lane_off + C::kColO + mt * D;
        const uint64_t scale2 = ttk::f2_pack(g.scale_log2, g.scale_log2);
        float* my_x = xchg + (mt * 2 + half) * 128 + lane_row;
        const float* other_x = xchg + (mt * 2 + (half ^ 1)) * 128 + lane_row;
        const int bar_id = 1 + mt;  // named barrier of this tile's two halves
        float m_run = -CUDART_INF_F;
        float l_part = 0.f;  // sum of p over this half's keys
        // keys of round j at or past lim lie outside: S on the block's round, else the
        // context end less the round's first key
        const int lim_ctx = ctx - (t0 - nblk) * kTileKeys;
        for (int j = 0; j < nt; ++j) {
            // A wait that runs out is recorded, but the loop goes on: every thread of
            // the tile must reach the named barriers below the same number of times.
            // (After a missed phase the later parity waits return at once.)
            if (!ttk::mbar_wait(sfull_bar(mt), (uint32_t)(j & 1))) ok = false;
            ttk::tc_fence_after();
            const int lim = (j < nblk) ? g.S : lim_ctx - j * kTileKeys;
            const int k0 = 64 * half;  // first key of this half
            float rmax = -CUDART_INF_F;
            {
                uint32_t a0[32], a1[32];
                ttk::tmem_ld32(tS + k0, a0);
                ttk::tmem_ld32(tS + k0 + 32, a1);
                ttk::tmem_ld_wait32(a0);
                tie32(a1);
                float r0 = -CUDART_INF_F, r1 = -CUDART_INF_F;
                if (lim >= kTileKeys) {
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        r0 = ttk::fmax3(r0, __uint_as_float(a0[c]), __uint_as_float(a0[c + 1]));
                        r1 = ttk::fmax3(r1, __uint_as_float(a1[c]), __uint_as_float(a1[c + 1]));
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        r0 = fmaxf(r0, (k0 + c < lim) ? __uint_as_float(a0[c]) : -CUDART_INF_F);
                        r1 = fmaxf(r1, (k0 + 32 + c < lim) ? __uint_as_float(a1[c]) : -CUDART_INF_F);
                    }
                }
                rmax = fmaxf(r0, r1);
            }
            // Row max of the raw scores over both halves (scale > 0 commutes with it).
            *my_x = rmax;
            ttk::tc_fence_before();
            named_sync(bar_id, 256);
            ttk::tc_fence_after();
            const float mx = fmaxf(*my_x, *other_x) * g.scale_log2;
            if (j == 0) {
                m_run = mx;
            } else {
                const bool need = mx > m_run + kRescaleThreshold;
                if (__any_sync(0xffffffffu, need)) {
                    // O is stable here: PV(mt, j-1) completed before QK(mt, j).  Each
                    // half rescales its D/2 columns of the row.
                    const float alpha = need ? exp2f(m_run - mx) : 1.0f;
                    if (need) {
                        m_run = mx;
                        l_part *= alpha;
                    }
#pragma unroll
                    for (int cc = 0; cc < D / 2; cc += 32) {
                        uint32_t o[32];
                        ttk::tmem_ld32(tO + half * (D / 2) + cc, o);
                        ttk::tmem_ld_wait32(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        ttk::tmem_st32(tO + half * (D / 2) + cc, o);
                    }
                }
            }
            // p = 2^(s*scale*log2e - m), 32 keys at a time re-read from TMEM: one packed
            // FMA per pair, then the SFU.  P (bf16 pairs) goes over the front of this
            // half's own 64 S columns, which only this thread reads.  The row sum adds
            // the unrounded p.
            const uint64_t negm2 = ttk::f2_pack(-m_run, -m_run);
            uint64_t lsum2 = ttk::f2_pack(0.f, 0.f);
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t a[32];
                ttk::tmem_ld32(tS + k0 + 32 * c2, a);
                ttk::tmem_ld_wait32(a);
                if (lim < kTileKeys) {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (k0 + 32 * c2 + c >= lim) a[c] = __float_as_uint(-CUDART_INF_F);
                }
                uint32_t pw[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint64_t e2 = ttk::f2_fma(ttk::f2_pack(__uint_as_float(a[2 * c]), __uint_as_float(a[2 * c + 1])),
                                                    scale2, negm2);
                    float e0, e1;
                    ttk::f2_unpack(e2, e0, e1);
                    const float p0 = ttk::ex2_ftz(e0), p1 = ttk::ex2_ftz(e1);
                    const __nv_bfloat162 pr = __floats2bfloat162_rn(p0, p1);
                    pw[c] = *reinterpret_cast<const uint32_t*>(&pr);
                    lsum2 = ttk::f2_add(lsum2, ttk::f2_pack(p0, p1));
                }
                ttk::tmem_st16(tS + k0 + 16 * c2, pw);
            }
            {
                float x0, x1;
                ttk::f2_unpack(lsum2, x0, x1);
                l_part += x0 + x1;
            }
            if (q == 0 && lim < kTileKeys) {
                // Last tile of a key range that ends inside it: the V rows past the end
                // hold whatever the cache has there.  P is 0 for them, but 0 * NaN
                // would still poison O, so zero those rows before PV(0, j) reads them
                // (PV(1, j) is issued after PV(0, j)).  K and V of this tile have
                // landed: QK(0, j) has completed.
                uint8_t* vst = smem + C::kRing + (size_t)(j % NS) * C::kStage + C::kTile;
                constexpr int kChunks = NP * 8;  // 16-byte chunks per V row
                for (int i2 = lane_row; i2 < (kTileKeys - lim) * kChunks; i2 += 128) {
                    const int key = lim + i2 / kChunks;
                    const int ch = i2 % kChunks;
                    *reinterpret_cast<uint4*>(vst + (ch >> 3) * C::kPart + key * 128 + ((ch & 7) << 4)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                ttk::fence_proxy_async_smem();
            }
            ttk::tmem_st_wait();
            ttk::tc_fence_before();
            ttk::mbar_arrive(pfull_bar(mt));
        }
        if (ok) ok = ttk::mbar_wait(ofull_bar, 0);
        // The row's l: this half's sum plus the other half's (same m for both).
        float* my_l = xchg + (mt * 2 + half) * 128 + lane_row;
        const float* other_l = xchg + (mt * 2 + (half ^ 1)) * 128 + lane_row;
        named_sync(bar_id, 256);  // every read of the max slots is done
        *my_l = ok ? l_part : 0.f;
        named_sync(bar_id, 256);
        const float l = l_part + *other_l;
        if (!ok && lane_row == 0 && half == 0) ttk::report_error(p.err, ttk::kErrTimeout);
        // The tensor-store epilogue is chosen the same way by every thread of the CTA,
        // and every thread of a tile goes through its named barrier whether or not its
        // waits ran out (a partial state that ran out is marked empty instead).
        if (!direct && g.fused) {
            fused_combine<D>(p, tO, half, row_valid, r_glob, b, gkv, rg, split, nv, n_mt, ok, m_run, l, q, lane_row,
                             tid, reinterpret_cast<volatile int*>(smem + C::kSlot + 8));
        } else if (direct ? maps.out_tma != 0 : true) {
            // Epilogue: this half's D/2 columns of the O row go TMEM -> registers ->
            // 128-row x 128-byte boxes in shared memory (128-byte swizzle, so a warp's
            // stores of 32 rows fall in different banks; the Q tiles and the K/V ring
            // are idle once every MMA has completed) -> tensor stores issued by one
            // thread, whose maps clip rows past R (partials) or past the block's S
            // positions (output).  Single split: normalised bf16 output; otherwise the
            // fp32 partial accumulator.
            ttk::tc_fence_after();
            constexpr int kNbF = D / 32;  // fp32 boxes per row
            constexpr int kNbH = D / 64;  // bf16 boxes per row
            const int nb = direct ? kNbH : kNbF;
            uint8_t* tile_base = smem + (size_t)mt * nb * 16384;
            const float inv = 1.0f / l;
#pragma unroll
            for (int cc = 0; cc < D / 2; cc += 32) {
                uint32_t o[32];
                ttk::tmem_ld32(tO + half * (D / 2) + cc, o);  // warp-collective: every lane loads
                ttk::tmem_ld_wait32(o);
                if (direct) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {  // 8 bf16 = one 16-byte chunk
                        uint32_t w[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const __nv_bfloat162 pr = __floats2bfloat162_rn(
                                __uint_as_float(o[8 * e + 2 * u]) * inv, __uint_as_float(o[8 * e + 2 * u + 1]) * inv);
                            w[u] = *reinterpret_cast<const uint32_t*>(&pr);
                        }
                        const int chunk = (half * (D / 2) + cc + 8 * e) / 8;
                        uint8_t* dst = tile_base + (chunk >> 3) * 16384 + lane_row * 128 +
                                       (((chunk & 7) ^ (lane_row & 7)) << 4);
                        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {  // 4 fp32 = one 16-byte chunk
                        const int chunk = (half * (D / 2) + cc + 4 * e) / 4;
                        uint8_t* dst = tile_base + (chunk >> 3) * 16384 + lane_row * 128 +
                                       (((chunk & 7) ^ (lane_row & 7)) << 4);
                        *reinterpret_cast<uint4*>(dst) = make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
                    }
                }
            }
            ttk::fence_proxy_async_smem();
            named_sync(3, 256 * n_mt);  // every row of every tile is staged
            if (q == 0 && lane_row == 0) {
                for (int t = 0; t < n_mt; ++t) {
                    const int row0 = rg * g.rows_per_cta + t * 128;
                    for (int bx = 0; bx < nb; ++bx) {
                        const uint32_t src = ttk::smem_u32(smem + (size_t)(t * nb + bx) * 16384);
                        if (direct)
                            ttk::tma_store_4d(&maps.out, src, bx * 64, gkv * g.G, row0 / g.G, b);
                        else
                            ttk::tma_store_3d(&maps.part, src, bx * 32, row0,
                                              (b * g.Hkv + gkv) * g.n_splits + split);
                    }
                }
                ttk::bulk_commit();
                ttk::bulk_wait_read();  // shared memory may be released; the writes land on their own
            }
            if (row_valid && half == 0) {
                if (direct) {
                    if (p.lse != nullptr) {
                        const int s = r_glob / g.G, jh = r_glob % g.G;
                        p.lse[((size_t)b * g.S + s) * g.Hq + (size_t)gkv * g.G + jh] = (m_run + log2f(l)) * kLn2;
                    }
                } else {
                    const size_t pi = ((size_t)(b * g.Hkv + gkv) * g.n_splits + split) * (size_t)g.R + r_glob;
                    p.part_ml[2 * pi + 0] = ok ? m_run : -CUDART_INF_F;
                    p.part_ml[2 * pi + 1] = ok ? l : 0.f;
                }
            }
        } else if (ok) {
            // Single split with G not dividing 128 (no box covers whole positions):
            // each half row goes TMEM -> registers -> shared memory -> one bulk copy.
            // A row stride of D*2 + 16 bytes keeps the 16-byte stores of consecutive
            // rows in different banks.
            ttk::tc_fence_after();
            uint8_t* hrow = smem + (size_t)(r_local * 2 + half) * C::kHalfRow;
            const float inv = 1.0f / l;
#pragma unroll
            for (int cc = 0; cc < D / 2; cc += 32) {
                uint32_t o[32];
                ttk::tmem_ld32(tO + half * (D / 2) + cc, o);  // warp-collective: every lane loads
                ttk::tmem_ld_wait32(o);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t w[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const __nv_bfloat162 pr = __floats2bfloat162_rn(
                            __uint_as_float(o[8 * e + 2 * u]) * inv, __uint_as_float(o[8 * e + 2 * u + 1]) * inv);
                        w[u] = *reinterpret_cast<const uint32_t*>(&pr);
                    }
                    *reinterpret_cast<uint4*>(hrow + (cc + 8 * e) * 2) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            if (row_valid) {
                ttk::fence_proxy_async_smem();
                const int s = r_glob / g.G, jh = r_glob % g.G;
                const size_t orow = ((size_t)b * g.S + s) * g.Hq + (size_t)gkv * g.G + jh;
                ttk::bulk_store(p.out + orow * D + half * (D / 2), ttk::smem_u32(hrow), D);
                ttk::bulk_commit();
                if (half == 0 && p.lse != nullptr) p.lse[orow] = (m_run + log2f(l)) * kLn2;
                ttk::bulk_wait_read();  // shared memory may be released; the writes land on their own
            }
        }
    }

    // TMEM is released only after every MMA this CTA issued has completed (the
    // issuing lane waited for that above).
    ttk::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ttk::tc_fence_after();
        ttk::tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------------
// Combine: partial states of the context splits -> out, lse.  One warp per output
// row (b, s, h); lanes hold D/32 columns each.  Every split's (m, l) pair and the
// lane's accumulator slice are requested together, four or eight splits per round
// trip (the pass is latency-bound: a few hundred bytes per row, so with at most four
// splits the smaller batch's registers leave room for more rows in flight per SM),
// and folded into a running (max, sum, accumulator) as they arrive.  When the prep
// kernel chose the split length, the grid is one resident wave striding over the rows:
// most calls then have few or no split row groups, and the wave exits at once.
// ---------------------------------------------------------------------------------
template <int D, int kBatch>
__device__ __forceinline__ void merge_row(const AttnMergeParams& p, long long row, int tps) {
    constexpr int PER = D / 32;  // kBatch: splits requested together (4 or 8)
    const AttnGeom& g = p.g;
    const int lane = threadIdx.x & 31;
    const int h = (int)(row % g.Hq);
    const int s = (int)((row / g.Hq) % g.S);
    const int b = (int)(row / ((long long)g.Hq * g.S));
    if (p.skip_if_zero != nullptr && __ldg(p.skip_if_zero + b) == 0) return;
    const int gkv = h / g.G, j = h % g.G;
    const int cap = g.page_size ? g.max_pages * g.page_size : g.max_ctx;
    int ctx = p.ctx_len ? __ldg(p.ctx_len + b) : g.max_ctx;
    if (ctx < 0 || ctx > cap) ctx = 0;  // reported by the split pass
    const int n_tiles = (ctx + kTileKeys - 1) / kTileKeys;
    // Split 0 always holds the block's keys; the others hold context tiles.  A row group
    // with one non-empty split was written by the split pass directly.
    const int n_valid = max(1, (n_tiles + tps - 1) / tps);
    if (n_valid == 1) return;
    const size_t base = ((size_t)(b * g.Hkv + gkv) * g.n_splits) * (size_t)g.R + (size_t)(s * g.G + j);

    float m = -CUDART_INF_F, lsum = 0.f;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    for (int c0 = 0; c0 < n_valid; c0 += kBatch) {
        const int nc = min(kBatch, n_valid - c0);
        float mc[kBatch], lc[kBatch], a[kBatch][PER];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int cu = c0 + min(u, nc - 1);  // in range; repeats beyond nc are not used
            const size_t pi = base + (size_t)cu * g.R;
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + pi);
            mc[u] = ml.x;
            lc[u] = ml.y;
            const float* ap = p.part_acc + pi * D + lane * PER;
            if (PER == 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(ap));
                a[u][0] = v.x; a[u][1 % PER] = v.y; a[u][2 % PER] = v.z; a[u][3 % PER] = v.w;
            } else {
                const float2 v = __ldcg(reinterpret_cast<const float2*>(ap));
                a[u][0] = v.x; a[u][1 % PER] = v.y;
            }
        }
        // an empty partial state (m = -inf) carries no weight; its accumulator was
        // never written and is not used
        float mn = m;
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (u < nc) mn = fmaxf(mn, mc[u]);
        if (mn == -CUDART_INF_F) continue;
        if (m != -CUDART_INF_F && mn != m) {
            const float r = exp2f(m - mn);
            lsum *= r;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] *= r;
        }
        m = mn;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (u >= nc || mc[u] == -CUDART_INF_F) continue;
            const float w = exp2f(mc[u] - m);
            lsum = fmaf(w, lc[u], lsum);
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, a[u][e], acc[e]);
        }
    }
    const float inv = 1.0f / lsum;
    const size_t orow = ((size_t)b * g.S + s) * g.Hq + h;
    uint16_t* op = p.out + orow * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; e += 2) {
        const __nv_bfloat162 pr = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
        *reinterpret_cast<uint32_t*>(op + e) = *reinterpret_cast<const uint32_t*>(&pr);
    }
    if (p.lse != nullptr && lane == 0) p.lse[orow] = (m + log2f(lsum)) * kLn2;
}

template <int D, int kBatch>
__global__ void __launch_bounds__(256) attn_merge_kernel(const __grid_constant__ AttnMergeParams p) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    const AttnGeom& g = p.g;
    int tps = g.tiles_per_split;
    if (p.order != nullptr) {
        const long long n_units = (long long)g.B * g.Hkv * g.n_rg * g.n_splits;
        if (__ldg(p.order + n_units + 2) == 0) return;  // this call split no row group
        tps = __ldg(p.order + n_units + 1);
    }
    const long long rows = (long long)g.B * g.S * g.Hq;
    const long long stride = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += stride)
        merge_row<D, kBatch>(p, row, tps);
}

// Work units of a ragged batch, sorted by their number of key tiles, longest first (a
// counting sort in one CTA; the hardware then dispatches the long units first and the
// grid's tail is short).  A unit's length is the split's context tiles plus the
// block's own keys on split 0; sequences that are skipped or finished have none.
// With lpt_dyn the split length is chosen here, per call, from the active sequences:
// tiles_per_split times 1, 2, 4, ... (at most the longest context), by an estimate of
// the span in tile-times: max(longest unit, total / SMs) + ~4 tiles of pipeline fill
// per wave of CTAs + ~32 tiles when anything is split (partial states and the combine
// pass; fitted to the ragged paged batch: one split 459 us, units of the per-SM share
// 466 us, two splits 497 us).  A block's first step (every sequence active) then takes
// whole row groups and no combine; later steps, with a few long sequences left, cut
// them into 64-tile units.
// Output: order[0 .. count) units, order[n_units] = count, order[n_units + 1] = split
// length, order[n_units + 2] = 1 if some row group has more than one split.
constexpr int kOrderThreads = 1024;
constexpr int kOrderCands = 8;     // split lengths tried: tiles_per_split << 0 .. 7
constexpr int kOrderCache = 4096;  // items whose tile counts stay in shared memory
__global__ void __launch_bounds__(kOrderThreads) attn_order_kernel(const __grid_constant__ AttnSplitParams p) {
    ttk::pdl_wait();
    ttk::pdl_trigger();
    __shared__ int hist[kOrderMaxLen + 1];
    __shared__ int s_tiles[kOrderCache];
    __shared__ unsigned s_total, s_lmax, s_active, s_units[kOrderCands];
    __shared__ int s_tps, s_split;
    const AttnGeom& g = p.g;
    const int n_items = g.B * g.Hkv * g.n_rg;
    const int n_units = n_items * g.n_splits;
    const int cap = g.page_size ? g.max_pages * g.page_size : g.max_ctx;
    const int base = g.tiles_per_split;
    const bool cached = n_items <= kOrderCache;
    const int lane = threadIdx.x & 31;
    int32_t* order = const_cast<int32_t*>(p.order);
    // context tiles of an item's sequence, or -1 when it takes no part in this call
    auto item_tiles = [&](int item) -> int {
        const int b = item / (g.n_rg * g.Hkv);
        const int keep = p.skip_if_zero != nullptr ? __ldg(p.skip_if_zero + b) : 1;
        const int ctx = p.ctx_len ? __ldg(p.ctx_len + b) : g.max_ctx;
        if (keep == 0) return -1;
        if (ctx < 0 || ctx > cap) return 0;  // split 0 alone: the split pass reports it
        return (ctx + kTileKeys - 1) / kTileKeys;
    };
    for (int i = threadIdx.x; i <= kOrderMaxLen; i += kOrderThreads) hist[i] = 0;
    if (threadIdx.x == 0) {
        s_total = 0;
        s_lmax = 0;
        s_active = 0;
        for (int c = 0; c < kOrderCands; ++c) s_units[c] = 0;
    }
    __syncthreads();
    // Sums over the items (each below 2^31: at most kOrderMaxUnits items of at most
    // kOrderMaxLen tiles), reduced per warp, one shared atomic per warp and sum; the
    // tile counts are kept for the two passes over the units.
    unsigned tot = 0, lmax = 0, active = 0, units[kOrderCands] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int it = threadIdx.x; it < ((cached || g.lpt_dyn) ? n_items : 0); it += kOrderThreads) {
        const int L = item_tiles(it);
        if (cached) s_tiles[it] = L;
        if (L < 0 || !g.lpt_dyn) continue;
        ++active;
        tot += (unsigned)L + 1u;
        lmax = max(lmax, (unsigned)L);
#pragma unroll
        for (int c = 0; c < kOrderCands; ++c) units[c] += (unsigned)max(1, (L + (base << c) - 1) / (base << c));
    }
    if (g.lpt_dyn) {
        tot = __reduce_add_sync(0xffffffffu, tot);
        lmax = __reduce_max_sync(0xffffffffu, lmax);
        active = __reduce_add_sync(0xffffffffu, active);
#pragma unroll
        for (int c = 0; c < kOrderCands; ++c) units[c] = __reduce_add_sync(0xffffffffu, units[c]);
        if (lane == 0 && active != 0) {
            atomicAdd(&s_total, tot);
            atomicMax(&s_lmax, lmax);
            atomicAdd(&s_active, active);
#pragma unroll
            for (int c = 0; c < kOrderCands; ++c) atomicAdd(&s_units[c], units[c]);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            const long long n_active = (long long)s_active;
            const long long share = ((long long)s_total + 147) / 148;
            long long best = -1;
            int best_c = 0;
            for (int c = 0; c < kOrderCands; ++c) {
                const long long t = (long long)base << c;
                if (c > 0 && ((long long)base << (c - 1)) >= s_lmax) break;  // longer splits change nothing
                const long long longest = (t < (long long)s_lmax ? t : (long long)s_lmax) + 1;
                const long long waves = ((long long)s_units[c] + 147) / 148;
                const bool split = (long long)s_units[c] > n_active;
                const long long est = max(longest, share) + 4 * waves + (split ? 32 : 0);
                if (best < 0 || est <= best) {
                    best = est;
                    best_c = c;
                }
            }
            s_tps = base << best_c;
            s_split = (long long)s_units[best_c] > n_active ? 1 : 0;
        }
    } else if (threadIdx.x == 0) {
        s_tps = base;
        s_split = g.n_splits > 1 ? 1 : 0;
    }
    __syncthreads();
    const int tps = s_tps;
    // Length class of unit u (0: empty).  Units are walked in whole-warp steps and the
    // lanes of one class share one shared-memory atomic: most units of a split batch
    // have the same length, and one atomic per unit would queue on that counter.
    auto unit_class = [&](int u) -> int {
        if (u >= n_units) return 0;
        const int item = u % n_items, split = u / n_items;
        const int L = cached ? s_tiles[item] : item_tiles(item);
        if (L < 0) return 0;
        const int t0 = split * tps;
        const int t1 = min(L, t0 + tps);
        return min((split == 0 ? 1 : 0) + max(0, t1 - t0), kOrderMaxLen);
    };
    for (int u0 = 0; u0 < n_units; u0 += kOrderThreads) {
        const int cls = unit_class(u0 + (int)threadIdx.x);
        const unsigned peers = __match_any_sync(0xffffffffu, cls);
        if (cls > 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[cls], __popc(peers));
    }
    __syncthreads();
    {
        // start of each length's slots, longest first: thread t holds length
        // kOrderMaxLen - t, an exclusive scan over the block (warp scans, then the warp
        // totals)
        static_assert(kOrderThreads == kOrderMaxLen, "one length per thread");
        __shared__ int wsum[kOrderThreads / 32];
        const int t = threadIdx.x, warp = t >> 5;
        const int len = kOrderMaxLen - t;
        const int c = hist[len];
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += v;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        const int start = (warp > 0 ? wsum[warp - 1] : 0) + incl - c;
        hist[len] = start;
        if (t == kOrderThreads - 1) {
            order[n_units] = start + c;
            order[n_units + 1] = tps;
            order[n_units + 2] = s_split;
        }
    }
    __syncthreads();
    for (int u0 = 0; u0 < n_units; u0 += kOrderThreads) {
        const int u = u0 + (int)threadIdx.x;
        const int cls = unit_class(u);
        const unsigned peers = __match_any_sync(0xffffffffu, cls);
        const int leader = __ffs(peers) - 1;
        int slot = 0;
        if (cls > 0 && lane == leader) slot = atomicAdd(&hist[cls], __popc(peers));
        slot = __shfl_sync(0xffffffffu, slot, leader) + __popc(peers & ((1u << lane) - 1u));
        if (cls > 0) order[slot] = u;
    }
}

// Modelled cost, in quarter tile-times, of splitting every (sequence, kv head, row
// group) item's n_tiles context tiles into `splits` ranges: waves of one CTA per SM,
// each paying its tiles plus ~3 tiles of set-up, pipeline fill and epilogue; the merge's
// serial depth (8 partial states in flight per round); and the partial-state traffic.
long long split_cost(long long items, int n_tiles, int splits) {
    const long long ctas = items * splits;
    const long long waves = (ctas + 147) / 148;
    const long long tps = (n_tiles + splits - 1) / splits;
    return 4 * waves * (tps + 3) + 4 * ((splits + 7) / 8) + (2 * ctas) / 148;
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
    if (Hkv > 65535 || B > 65535) { *why = "B and Hkv must be at most 65535"; return false; }
    g.R = g.G * S;
    g.rows_per_cta = g.R < 256 ? g.R : 256;
    g.n_rg = (g.R + 255) / 256;
    g.n_mt = (g.rows_per_cta + 127) / 128;
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
    if (g.R > 128 && (long long)B * Hkv * g.n_rg * (n_tiles + 1) <= 148LL * 8) {
        // A problem of a few 128-key rounds per SM in all is latency-bound: one 128-row
        // tile per CTA halves each round's tensor work and doubles the CTAs (the second
        // row tile's CTA finds the same K/V tiles in L2).
        g.rows_per_cta = 128;
        g.n_rg = (g.R + 127) / 128;
        g.n_mt = 1;
    }
    const long long items = (long long)B * Hkv * g.n_rg;
    int tps;
    bool dyn = false;
    if (num_splits > 0) {
        tps = n_tiles > 0 ? (n_tiles + num_splits - 1) / num_splits : 1;
    } else if (n_tiles == 0) {
        tps = 1;
    } else {
        int best = 1;
        long long best_cost = split_cost(items, n_tiles, 1);
        const int max_s = n_tiles < 1024 ? n_tiles : 1024;
        for (int s = 2; s <= max_s; ++s) {
            const long long c = split_cost(items, n_tiles, s);
            if (c < best_cost) { best_cost = c; best = s; }
        }
        tps = (n_tiles + best - 1) / best;
        if (page_size != 0 && items > 148 && n_tiles + 1 <= kOrderMaxLen) {
            // A ragged paged batch of several waves: the prep kernel picks the split
            // length per call (this one times 1, 2, 4, ...) from the sequences that are
            // active, and the units go out longest first.  The finest length is 64
            // tiles, or an eighth of the longest context if that is longer.
            tps = max(64, (n_tiles + 7) / 8);
            if (tps > n_tiles) tps = n_tiles;
            dyn = true;
        } else if (page_size != 0 && tps < 64 && n_tiles > 64) {
            // shorter sequences of a paged batch leave their later splits empty (those
            // CTAs exit at once), so keep splits long enough to amortise a CTA
            tps = 64;
        }
    }
    if (tps < 1) tps = 1;
    g.tiles_per_split = tps;
    g.n_splits = n_tiles > 0 ? (n_tiles + tps - 1) / tps : 1;
    if (g.n_splits > 65535) { *why = "too many context splits"; return false; }
    if ((long long)B * Hkv * g.n_rg * g.n_splits > 0x7fffffffLL) { *why = "too many work units"; return false; }
    // Ragged batches spanning several waves: units dispatched longest first.  The sort
    // is a counting sort over lengths of at most tiles_per_split + 1 tiles.
    g.lpt = (page_size != 0 && (long long)B * Hkv * g.n_rg * g.n_splits > 148 && tps + 1 <= kOrderMaxLen &&
             (long long)B * Hkv * g.n_rg * g.n_splits <= kOrderMaxUnits) ? 1 : 0;
    g.lpt_dyn = (g.lpt && dyn) ? 1 : 0;
    g.fused = 0;  // the caller decides (it needs the device's SM count)
    return true;
}

// Workspace: fp32 partial accumulators [B][Hkv][n_splits][R][D], then (m, l) pairs,
// then two counters per row group (the combine inside the split pass; zero on entry,
// left at zero), then (ragged batches) the work order: units + 3 words.
void attn_layout(const AttnGeom& g, void* ws, float** part_acc, float** part_ml, unsigned** ticket,
                 int32_t** order) {
    const size_t rows = (size_t)g.B * g.Hkv * g.n_splits * g.R;
    size_t acc = (rows * g.D * sizeof(float) + 255) & ~size_t(255);
    size_t ml = (rows * 2 * sizeof(float) + 255) & ~size_t(255);
    size_t tk = (2 * (size_t)g.B * g.Hkv * g.n_rg * sizeof(unsigned) + 255) & ~size_t(255);
    char* w = static_cast<char*>(ws);
    *part_acc = reinterpret_cast<float*>(w);
    *part_ml = reinterpret_cast<float*>(w + acc);
    *ticket = reinterpret_cast<unsigned*>(w + acc + ml);
    *order = g.lpt ? reinterpret_cast<int32_t*>(w + acc + ml + tk) : nullptr;
}

size_t attn_workspace_bytes(const AttnGeom& g) {
    const size_t rows = (size_t)g.B * g.Hkv * g.n_splits * g.R;
    size_t acc = (rows * g.D * sizeof(float) + 255) & ~size_t(255);
    size_t ml = (rows * 2 * sizeof(float) + 255) & ~size_t(255);
    size_t tk = (2 * (size_t)g.B * g.Hkv * g.n_rg * sizeof(unsigned) + 255) & ~size_t(255);
    const size_t units = (size_t)g.B * g.Hkv * g.n_rg * g.n_splits;
    return acc + ml + tk + (g.lpt ? (units + 3) * sizeof(int32_t) : 0) + 256;
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
                                 (int)Cfg<128>::kBytes);
    else
        e = cudaFuncSetAttribute(attn_split_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)Cfg<64>::kBytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done |= (1ull << dev);
    return e;
}

cudaError_t launch_attn_order(const AttnSplitParams& p, cudaStream_t stream) {
    return launch_pdl(attn_order_kernel, dim3(1), dim3(kOrderThreads), 0, stream, p);
}

cudaError_t launch_attn_split(const AttnSplitParams& p, const AttnMaps& maps, cudaStream_t stream) {
    const AttnGeom& g = p.g;
    const unsigned n_items = (unsigned)(g.B * g.Hkv * g.n_rg);
    dim3 grid = p.order ? dim3(n_items * (unsigned)g.n_splits, 1, 1) : dim3(n_items, (unsigned)g.n_splits, 1);
    if (g.fused) {
        // the CTAs of a row group wait for one another: a cooperative launch keeps
        // every CTA resident (the caller checked that the grid fits one wave)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = g.D == 128 ? Cfg<128>::kBytes : Cfg<64>::kBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeCooperative;
        attr[1].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return g.D == 128 ? cudaLaunchKernelEx(&cfg, attn_split_kernel<128>, p, maps)
                          : cudaLaunchKernelEx(&cfg, attn_split_kernel<64>, p, maps);
    }
    if (g.D == 128)
        return launch_pdl(attn_split_kernel<128>, grid, dim3(kThreads), Cfg<128>::kBytes, stream, p, maps);
    else
        return launch_pdl(attn_split_kernel<64>, grid, dim3(kThreads), Cfg<64>::kBytes, stream, p, maps);
}

cudaError_t launch_attn_merge(const AttnMergeParams& p, cudaStream_t stream) {
    const AttnGeom& g = p.g;
    const long long rows = (long long)g.B * g.S * g.Hq;
    long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (p.order != nullptr && blocks > 148 * 4) blocks = 148 * 4;  // one resident wave
    const bool few = g.n_splits <= 4;
    if (g.D == 128)
        return few ? launch_pdl(attn_merge_kernel<128, 4>, dim3((unsigned)blocks), dim3(256), 0, stream, p)
                   : launch_pdl(attn_merge_kernel<128, 8>, dim3((unsigned)blocks), dim3(256), 0, stream, p);
    else
        return few ? launch_pdl(attn_merge_kernel<64, 4>, dim3((unsigned)blocks), dim3(256), 0, stream, p)
                   : launch_pdl(attn_merge_kernel<64, 8>, dim3((unsigned)blocks), dim3(256), 0, stream, p);
}

}  // namespace tti
