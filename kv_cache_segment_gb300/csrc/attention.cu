// attention.cu -- the persistent Multi-Segment Attention kernel for sm_103a.
//
// One launch serves every work item of a plan: decode groups (a sequence's
// few trailing query rows, all G query heads of one kv head packed as the
// rows of a warp-level MMA) and prefill / hole-recompute items (two query
// tiles of 128 rows x one head that share a kv head -- two heads over the
// same rows, or for an odd Hq/Hkv one head over two consecutive row tiles --
// on the tcgen05 tensor cores with TMEM accumulators).  KV tiles are 128-key
// windows of an item's logical key range; the producer fetches each window
// from the physically contiguous segments it overlaps, in TMA boxes of 128,
// 64, 32 or 16 rows per piece (AsymCache
// explainer, "核心方法 1. Multi-Segment Attention": attention over the
// physically contiguous segments of the live KV; MSA summary: one kernel over
// many disjoint segments instead of a launch per segment).  Inside an item
// the online-softmax running (max, sum, output) state carries across
// segments, which is the pairwise form of the log-sum-exp merge; items of a
// group that was split for SM balance write (output, lse) partials and the
// last one to finish merges them by log-sum-exp.
//
// CTA roles, launch with prefill items (12 warps):
//   warp 0      K producer: takes the CTA's items (the first by position,
//               the rest from the global work queue), loads the Q tiles of
//               prefill items and the K tiles (TMA) into a ring of
//               shared-memory stages, records each tile's key range.
//   warp 1      owns TMEM; runs the MMA issue loop converged, one elected
//               lane issuing tcgen05.mma.  Per KV tile j, in this order:
//               PV0(j-1), S0(j), PV1(j-1), S1(j), where Sk = Qk K^T lands in
//               TMEM buffer k and PVk accumulates O_k += P_k V with P_k read
//               from TMEM (it overwrites S_k; the tensor core runs one
//               thread's MMAs in issue order).
//   warp 2      V producer: the V tiles, on a ring of their own.
//   warp 3      merge warp: finishes decode items (combines the compute
//               warps' states, writes out / partials, cross-CTA merge).
//   warps 4..7  warpgroup 0: softmax of Q tile 0 (thread = row = TMEM lane)
//               and the decode math (mma.sync, 32 keys per warp per tile).
//   warps 8..11 warpgroup 1: softmax of Q tile 1.
// Each softmax warpgroup has the other's PV + S (about 1024 tensor cycles) to
// produce its P before the tensor core needs it.
// Launch with decode items only (7 warps): K producer, V producer, the four
// decode warps, the merge warp.
#include <cuda.h>
#include <atomic>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>

#include "msa_internal.h"
#include "plan.h"
#include "ptx.cuh"

namespace msa {

struct AttnParams {
    const Item* items;
    const Group* groups;
    const Run* runs;
    const int32_t* pos;
    const int32_t* order;  // item ids, longest first (the dynamic queue)
    int32_t* sched;        // [0] queue head, [1] CTAs finished
    int32_t n_items;
    int32_t* counters;   // two per group: [2*group + head slot]
    int32_t* error_word;
    float* dec_part;
    float* dec_lse;
    float* pre_part;
    float* pre_lse;
    const __nv_bfloat16* q;
    void* out;
    float* lse;
    int32_t out_fp32;
    int32_t Hq;
    int32_t G;
    int32_t has_prefill;
    float scale_log2;
    int32_t n_runs;
    uint64_t limit_ns;
};

// Shared-memory plan of a CTA.  DEC = the launch has decode items only: no
// Q tiles, so those bytes become a third K/V stage (more bytes in flight for
// the HBM-bound path).  The decode merge scratch has its own region.
template <int D, bool DEC>
struct Cfg {
    // mixed launch: 3 warpgroups (producer/MMA, softmax 0, softmax 1) with
    // a register split; decode-only: producer + 4 compute warps
    static constexpr int kWarps = DEC ? 7 : 12;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kFirstCompute = DEC ? 2 : 4;  // first compute warp
    static constexpr int kComputeWarps = DEC ? 4 : 8;
    // combines the four compute warps' decode states and runs the cross-CTA
    // merge, so the compute warps go on to the next item at once
    static constexpr int kMergeWarp = DEC ? 6 : 3;
    static constexpr int kVWarp = DEC ? 1 : 2;          // the V-tile producer
    // Register split of the mixed launch (setmaxnreg): 384 threads launch with
    // 168 registers each (3 warps share an SM sub-partition's 16K registers);
    // warpgroup 0 gives back down to kRegsLow, the two softmax warpgroups grow
    // to kRegsHigh.  128*88 + 256*208 = 384*168 exactly.
    static constexpr int kRegsLaunch = 168;
    static constexpr int kRegsLow = 88;
    static constexpr int kRegsHigh = 208;
    static_assert(DEC || 128 * kRegsLow + 256 * kRegsHigh == kThreads * kRegsLaunch, "register split must balance");
    static constexpr int kPanels = D / 64;            // 64-element (128-byte) column panels
    static constexpr int kPanelBytes = 128 * 128;     // one panel of a 128-row tile
    static constexpr int kTileBytes = kPanels * kPanelBytes;  // 128 rows x D bf16
    static constexpr int kStages = DEC ? (D == 128 ? 3 : 6) : (D == 128 ? 2 : 4);
    static constexpr int kOffQ = 0;                   // Q tiles 0 and 1 (prefill)
    static constexpr int kOffK = DEC ? 0 : 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffScr = kOffV + kStages * kTileBytes;  // decode merge scratch [4][16][D] fp32
    static constexpr int kScrBytes = 4 * kDecRows * D * 4;
    static constexpr int kOffCtl = kOffScr + kScrBytes;
    static constexpr int kCtlBytes = 1536;
    static constexpr int kSmem = kOffCtl + kCtlBytes + 1024;  // + slack to align the base to 1024
    // TMEM: S buffers of 128 columns from column 0, then O0 and O1 (D columns
    // each).  At D = 128 that is S0, S1, O0, O1.  At D = 64 a third S buffer
    // fits, and the S MMAs rotate over the three (kRot): slot n of a CTA's
    // prefill work (tile j, query tile k, counted across items) uses buffer
    // n % 3, so the S of a query tile's next key tile is issued ahead of the
    // PV of its current one.
    static constexpr bool kRot = !DEC && D == 64;
    static constexpr int kSBufs = kRot ? 3 : 2;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmemO = kSBufs * 128;
    static_assert(kSmem + 64 <= 232448, "shared memory over the per-CTA limit");
    static_assert(kTmemO + 2 * D <= kTmemCols, "TMEM budget");
};

struct Ctl {
    uint64_t k_full[8], k_empty[8], v_full[8], v_empty[8];
    uint64_t q_full, q_empty;
    uint64_t s_full[3], p_full[3], p_empty[3];  // per S buffer
    uint64_t o_empty[2];
    uint64_t o_full;
    uint64_t drain;
    uint64_t csync[2];  // bounded barriers of warpgroup 0 / 1 (128 threads each)
    uint64_t item_full[4], item_empty[4];  // ring of item ids from the producer to the other roles
    uint64_t meta_full[8];  // tile metadata ring (K producer -> readers), slot = tile % 8
    int2 tmeta[8];          // per tile: first logical key, valid keys
    uint32_t tmem_base;
    int abort;
    int flag_last[2];
    int ring[4];
    float dec_m[4][kDecRows];
    float dec_l[4][kDecRows];
    float dec_lr[4][kDecRows];
    uint64_t merge_full, merge_empty;  // decode states in the scratch: compute warps <-> merge warp
    int merge_item;                    // item whose states are in the scratch (-1: no more)
};

static_assert(sizeof(Ctl) <= Cfg<128, false>::kCtlBytes, "control block too large");

constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ void fail(const AttnParams& p, Ctl* ctl, int code) {
    atomicOr(p.error_word, code);
    ctl->abort = 1;
}

__device__ __forceinline__ bool wait_bar(const AttnParams& p, Ctl* ctl, uint64_t* bar, uint32_t parity, int code) {
    if (ptx::mbar_wait(bar, parity, &ctl->abort, p.limit_ns)) return true;
    fail(p, ctl, code);
    return false;
}

// Query tile k (0 or 1) of a prefill group: two query heads of one kv head
// over the same <= 128 rows, or, for the last query head of a kv head when
// G is odd, consecutive 128-row tiles of that one head.  Either way both share the group's K/V tiles, so the two softmax
// warpgroups alternate on the tensor core.
// A group of more than 128 rows is always the second form; one of at most
// 128 rows has one tile in that form, where the two readings agree.
__device__ __forceinline__ bool qtile_rows_mode(const AttnParams& p, const Group& g) {
    return (p.G & 1) && g.nrows > kTileRows;
}
__device__ __forceinline__ int qtile_head(const AttnParams& p, const Group& g, int k) {
    return g.head + (qtile_rows_mode(p, g) ? 0 : k);
}
__device__ __forceinline__ int qtile_row0(const AttnParams& p, const Group& g, int k) {
    return g.row0 + (qtile_rows_mode(p, g) ? k * kTileRows : 0);
}
__device__ __forceinline__ int qtile_rows(const AttnParams& p, const Group& g, int k) {
    return qtile_rows_mode(p, g) ? min(kTileRows, g.nrows - k * kTileRows) : g.nrows;
}

// Sum of the two bf16 values packed in w, as fp32 (exact).
__device__ __forceinline__ float bf16x2_sum(uint32_t w) {
    return __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
}

// Barrier of one warpgroup (128 threads) built on an mbarrier, so that a
// wait that can never complete (a warp gave up on a timeout) runs out
// instead of hanging.  `cnt` counts this thread's passes.
__device__ __forceinline__ bool compute_sync(const AttnParams& p, Ctl* ctl, int wg, uint32_t& cnt) {
    ptx::mbar_arrive(&ctl->csync[wg]);
    const bool ok = wait_bar(p, ctl, &ctl->csync[wg], cnt & 1, kErrTimeoutCompute);
    ++cnt;
    return ok;
}

// Dynamic work queue.  The producer takes the next item id from a global
// counter over the longest-first order and passes it to the other roles of
// its CTA through a 4-deep shared ring (id -1 = no more work); every role
// therefore walks the same item sequence.
__device__ __forceinline__ int publish_item(const AttnParams& p, Ctl* ctl, uint32_t& n) {
    const int slot = n & 3;
    if (!wait_bar(p, ctl, &ctl->item_empty[slot], ((n >> 2) & 1) ^ 1, kErrTimeoutProducer)) return -2;
    // A CTA's first item is position blockIdx.x of the order (no queue
    // round trip before its first loads, and the longest items start on
    // distinct CTAs at once); later ones come from the global counter, which
    // hands out positions gridDim.x, gridDim.x + 1, ...
    const int q = n == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(&p.sched[0], 1);
    const int id = q < p.n_items ? p.order[q] : -1;
    ctl->ring[slot] = id;
    ptx::mbar_arrive(&ctl->item_full[slot]);
    ++n;
    return id;
}

__device__ __forceinline__ int take_item(const AttnParams& p, Ctl* ctl, uint32_t& n, int code) {
    const int slot = n & 3;
    if (!wait_bar(p, ctl, &ctl->item_full[slot], (n >> 2) & 1, code)) return -2;
    const int id = ctl->ring[slot];
    ptx::mbar_arrive(&ctl->item_empty[slot]);
    ++n;
    return id;
}

// Warp-wide forms for the MMA warp.  Every lane waits (each with acquire
// semantics, so each may then read what the barrier guards) and the warp
// votes, so it leaves converged with the same outcome everywhere.
__device__ __forceinline__ bool wait_bar_w(const AttnParams& p, Ctl* ctl, uint64_t* bar, uint32_t parity, int code) {
    const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, &ctl->abort, p.limit_ns));
    if (!ok) fail(p, ctl, code);
    return ok;
}

__device__ __forceinline__ int take_item_w(const AttnParams& p, Ctl* ctl, uint32_t& n, int code, int lane) {
    const int slot = n & 3;
    if (!wait_bar_w(p, ctl, &ctl->item_full[slot], (n >> 2) & 1, code)) return -2;
    const int id = ctl->ring[slot];
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&ctl->item_empty[slot]);  // one arrival per role
    ++n;
    return id;
}

// Byte offset of 16-byte chunk `c16` (0..D/8-1) of row `r` in a 128-row
// tile stored as 128-byte-swizzled 64-column panels (the TMA SWIZZLE_128B
// layout, which is also the tcgen05 canonical K-major layout).
template <int D>
__device__ __forceinline__ uint32_t sw128_off(int r, int c16) {
    const int panel = c16 >> 3, cc = c16 & 7;
    return (uint32_t)(panel * 16384 + r * 128 + ((cc ^ (r & 7)) << 4));
}

// ------------------------------------------------------------ producer --

// Two producer threads, one per ring: KSIDE (warp 0) takes items from the
// queue and publishes them, loads the Q tiles of prefill items and the K
// tiles, and records each tile's (first key, valid keys) in the metadata
// ring; the V side (its own warp) follows the same items and loads the V
// tiles.  The rings advance independently, so K for tile j+2 is fetched as
// soon as the S MMAs of tile j have read K(j), long before PV(j) frees V(j).
template <int D, bool DEC, bool KSIDE>
__device__ void producer(const AttnParams& p, uint8_t* smem, Ctl* ctl, const CUtensorMap* tm128,
                         const CUtensorMap* tm64, const CUtensorMap* tm32, const CUtensorMap* tm16,
                         const CUtensorMap* tmQ) {
    using C = Cfg<D, DEC>;
    uint64_t* full = KSIDE ? ctl->k_full : ctl->v_full;
    uint64_t* empty = KSIDE ? ctl->k_empty : ctl->v_empty;
    uint8_t* ring = smem + (KSIDE ? C::kOffK : C::kOffV);
    const int code = kErrTimeoutProducer;
    uint32_t kv_cnt = 0, q_cnt = 0, n_taken = 0;
    for (;;) {
        const int ii = KSIDE ? publish_item(p, ctl, n_taken) : take_item(p, ctl, n_taken, code);
        if (ii < 0) break;
        const Item it = p.items[ii];
        const Group g = p.groups[it.group];
        int kvh = g.head;
        if (KSIDE && DEC) {
            // The compute warps read this item's Q rows (G heads x D each,
            // contiguous per row) when they reach it, several tiles from now:
            // bring them into L2 first.  (Measured: +3 % in the decode-only
            // configuration, -2 % in the mixed one, where it is left out.)
            const uint32_t bytes = (uint32_t)(p.G * D * 2);
            for (int r = 0; r < g.nrows; ++r)
                ptx::prefetch_l2_bulk(static_cast<const __nv_bfloat16*>(p.q) +
                                          ((int64_t)(g.row0 + r) * p.Hq + (int64_t)g.head * p.G) * D,
                                      bytes);
        }
        if (!DEC && it.kind == kPrefill) {
            kvh = g.head / p.G;
            if (KSIDE) {
                const int nh = g.pad;  // query tiles of the item: 1 or 2 (see qtile_head)
                if (!wait_bar(p, ctl, &ctl->q_empty, (q_cnt & 1) ^ 1, code)) goto drain;
                ptx::mbar_arrive_expect_tx(&ctl->q_full, nh * C::kTileBytes);
                for (int k = 0; k < nh; ++k)
                    for (int pn = 0; pn < C::kPanels; ++pn)
                        ptx::tma_load_3d(smem + C::kOffQ + k * C::kTileBytes + pn * C::kPanelBytes, tmQ, pn * 64,
                                         qtile_head(p, g, k), qtile_row0(p, g, k), &ctl->q_full);
                ++q_cnt;
            }
        }
        {
            // KV tiles are 128-key windows of the item's logical key range.  A
            // window that lies inside one segment is one TMA rectangle; where it
            // spans segments, each piece is fetched from its own segment in
            // boxes of 64, 32 and 16 rows (segments are whole 16-row blocks, so
            // every piece is).
            int r = it.first_run;
            int tiles = 0;
            for (int t0 = it.kb; t0 < it.ke; t0 += kTileKeys) {
                if (tiles >= it.pad) {  // plan inconsistent: never run past the item
                    fail(p, ctl, kErrBadIndex);
                    goto drain;
                }
                ++tiles;
                const int t1 = min(t0 + kTileKeys, it.ke);
                const int n = t1 - t0;
                const int st = kv_cnt % C::kStages;
                const uint32_t ph = (kv_cnt / C::kStages) & 1;
                if (!wait_bar(p, ctl, &empty[st], ph ^ 1, code)) goto drain;
                if (KSIDE) {
                    ctl->tmeta[kv_cnt & 7] = make_int2(t0, n);
                    ptx::mbar_arrive(&ctl->meta_full[kv_cnt & 7]);
                }
                uint8_t* dst = ring + st * C::kTileBytes;
                ptx::mbar_arrive_expect_tx(&full[st], (uint32_t)(((n + kBlock - 1) & ~(kBlock - 1)) * D * 2));
                int cur = t0;
                while (cur < t1) {
                    if (r < 0 || r >= p.n_runs) {
                        fail(p, ctl, kErrBadIndex);
                        goto drain;
                    }
                    const Run R = p.runs[r];
                    const int rend = R.log_start + R.n_tok;
                    if (cur >= rend) { ++r; continue; }
                    const int pend = min(t1, rend);
                    const int phys = R.phys_row + (cur - R.log_start);
                    const int off = cur - t0;
                    if (off == 0 && pend - cur == kTileKeys) {
                        for (int pn = 0; pn < C::kPanels; ++pn)
                            ptx::tma_load_3d(dst + pn * C::kPanelBytes, tm128, pn * 64, kvh, phys, &full[st]);
                    } else {
                        // the piece's whole blocks, in boxes of 4, 2 or 1 blocks (64, 32, 16 rows)
                        const int nb = (pend - cur + kBlock - 1) / kBlock;
                        for (int b = 0; b < nb;) {
                            const int w = nb - b >= 4 ? 4 : (nb - b >= 2 ? 2 : 1);
                            const CUtensorMap* tm = w == 4 ? tm64 : (w == 2 ? tm32 : tm16);
                            for (int pn = 0; pn < C::kPanels; ++pn)
                                ptx::tma_load_3d(dst + pn * C::kPanelBytes + (off + b * kBlock) * 128, tm, pn * 64,
                                                 kvh, phys + b * kBlock, &full[st]);
                            b += w;
                        }
                    }
                    cur = pend;
                }
                ++kv_cnt;
            }
        }
    }
drain:
    // Wait (bounded, ignoring the abort flag) for the loads still in flight,
    // so that none lands in shared memory after the CTA has exited.
    {
        static __shared__ int never;  // an abort flag nobody sets
        never = 0;
        const uint32_t tail = kv_cnt < (uint32_t)C::kStages ? kv_cnt : (uint32_t)C::kStages;
        for (uint32_t k = kv_cnt - tail; k < kv_cnt; ++k)
            ptx::mbar_wait(&full[k % C::kStages], (k / C::kStages) & 1, &never, 100000000ull);
        if (KSIDE && q_cnt > 0) ptx::mbar_wait(&ctl->q_full, (q_cnt - 1) & 1, &never, 100000000ull);
    }
}

// ------------------------------------------------------------ MMA warp --

// The whole MMA warp runs this loop; elect.sync inside the MMA and commit
// instructions lets one lane issue.
template <int D, bool DEC>
__device__ void mma_issuer(const AttnParams& p, uint8_t* smem, Ctl* ctl, int lane) {
    using C = Cfg<D, DEC>;
    constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, 128, 0, 0);  // Q K-major, K K-major
    constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, D, 0, 1);   // P (TMEM), V MN-major
    const uint32_t tbase = ctl->tmem_base;
    // Shared-memory descriptors: the high word (stride 1024 bytes, version,
    // 128-byte swizzle) is common to every operand; the low words are built
    // once and advanced by byte offsets >> 4 added to their 14-bit address
    // field (every operand lies in this CTA's shared memory, < 256 KB, so
    // the field never carries over).  A single issuing thread needs a short
    // per-MMA instruction chain to keep up with the tensor pipe (64 cycles
    // per 128x128x16 MMA).
    const uint64_t dQ = ptx::smem_desc(ptx::smem_u32(smem + C::kOffQ), 16, 1024, 2);
    const uint32_t hi = (uint32_t)(dQ >> 32);
    const uint32_t lQ = (uint32_t)dQ;
    const uint32_t lK = (uint32_t)ptx::smem_desc(ptx::smem_u32(smem + C::kOffK), 16, 1024, 2);
    const uint32_t lV = (uint32_t)ptx::smem_desc(ptx::smem_u32(smem + C::kOffV), C::kPanelBytes, 1024, 2);
    // P-ready phases per query tile; O-free phases per query tile (tile 1's
    // barrier only moves in items that have a second tile)
    uint32_t kv_cnt = 0, q_cnt = 0, pf0 = 0, pf1 = 0, oc0 = 0, oc1 = 0, n_taken = 0;

    for (;;) {
        const int ii = take_item_w(p, ctl, n_taken, kErrTimeoutMma, lane);
        if (ii < 0) return;
        const Item it = p.items[ii];
        const int T = it.pad;  // KV tiles of this item
        if (it.kind != kPrefill) { kv_cnt += T; continue; }
        const Group g = p.groups[it.group];
        const int nh = g.pad;
        if (!wait_bar_w(p, ctl, &ctl->q_full, q_cnt & 1, kErrTimeoutMma)) return;
        ++q_cnt;
        int2 mt_prev = make_int2(0, 0);  // metadata of tile j-1, read when its S was issued
        for (int j = 0; j <= T; ++j) {
            const int jj = j - 1;
            const uint32_t kj = kv_cnt + j, kp = kv_cnt + jj;
            const int st = kj % C::kStages, stp = kp % C::kStages;
            const int nk = (mt_prev.y + 15) >> 4;
            int2 mt_cur = mt_prev;
            // V of tile j-1 and K of tile j first: they are normally loaded
            // long before, and waiting for them here keeps their waits off the
            // path from a warpgroup's P-ready signal to its next S
            if (j >= 1 && !wait_bar_w(p, ctl, &ctl->v_full[stp], (kp / C::kStages) & 1, kErrTimeoutMma)) return;
            if (j < T && !wait_bar_w(p, ctl, &ctl->k_full[st], (kj / C::kStages) & 1, kErrTimeoutMma)) return;
            for (int k = 0; k < nh; ++k) {
                // O_k += P_k V for tile j-1: P_k (bf16 pairs) read from TMEM
                // columns 0..63 of S_k (a softmax warp that needs the bf16
                // residual of its rows' P adds it itself before P is ready)
                if (j >= 1) {
                    if (!wait_bar_w(p, ctl, &ctl->p_full[k], (k ? pf1 : pf0) & 1, kErrTimeoutMma)) return;
                    if (k) ++pf1; else ++pf0;
                    if (jj == 0 &&
                        !wait_bar_w(p, ctl, &ctl->o_empty[k], ((k ? oc1 : oc0) & 1) ^ 1, kErrTimeoutMma))
                        return;
                    ptx::tc_fence_after();
                    const uint32_t vl = lV + (uint32_t)((stp * C::kTileBytes) >> 4);
                    const uint32_t to = tbase + C::kTmemO + k * D, tp = tbase + k * 128;
                    // 16 keys per MMA: V rows ks*16.. start 16*128 bytes further.
                    // O_k starts every item at zero (the softmax warpgroup
                    // clears it), so every PV MMA accumulates.
                    if (nk == kTileKeys / 16) {
#pragma unroll
                        for (int ks = 0; ks < kTileKeys / 16; ++ks)
                            ptx::tc_mma_ts_e<1>(to, tp + ks * 8, vl + ks * 128, hi, kIdescPV);
                    } else {
                        for (int ks = 0; ks < nk; ++ks) ptx::tc_mma_ts_e<1>(to, tp + ks * 8, vl + ks * 128, hi, kIdescPV);
                    }
                    ptx::tc_commit_e(&ctl->p_empty[k]);
                }
                // S_k = Q_k K^T for tile j
                if (j < T) {
                    if (k == 0) mt_cur = ctl->tmeta[kj & 7];
                    ptx::tc_fence_after();
                    const uint32_t kl = lK + (uint32_t)((st * C::kTileBytes) >> 4);
                    const uint32_t ql = lQ + (uint32_t)((k * C::kTileBytes) >> 4);
                    const uint32_t ts = tbase + k * 128;
                    // 16 dims per MMA: 32 bytes along a 128-byte swizzled row,
                    // the next 64 dims in the next panel
                    ptx::tc_mma_ss_e<0>(ts, ql, kl, hi, kIdescS);
#pragma unroll
                    for (int ks = 1; ks < D / 16; ++ks) {
                        const uint32_t off = (uint32_t)(((ks >> 2) * C::kPanelBytes + (ks & 3) * 32) >> 4);
                        ptx::tc_mma_ss_e<1>(ts, ql + off, kl + off, hi, kIdescS);
                    }
                    ptx::tc_commit_e(&ctl->s_full[k]);
                }
            }
            if (j >= 1) {
                ptx::tc_commit_e(&ctl->v_empty[stp]);
                if (jj == T - 1) {
                    ptx::tc_commit_e(&ctl->o_full);
                    ++oc0;
                    if (nh == 2) ++oc1;
                }
            }
            if (j < T) {
                ptx::tc_commit_e(&ctl->k_empty[st]);
                if (j == T - 1) ptx::tc_commit_e(&ctl->q_empty);
            }
            mt_prev = mt_cur;
        }
        kv_cnt += T;
    }
}

// MMA warp of the rotating-buffer launch (D = 64, three S buffers).  The
// prefill slots of the CTA, n = j * nh + k for key tile j and query tile k of
// an item, counted on across items, take S buffer n % 3.  The loop is the
// two-buffer one with the S MMA moved in front of the PV: as soon as query
// tile k's P of tile j-1 is ready, S_k(j) goes into the buffer that the PV
// of slot n - 3 (issued before it; the tensor pipe runs one thread's MMAs
// in order) has read, and only then PV_k(j-1).  A warpgroup's next S thus
// waits for its P-ready signal and four MMAs, not for twelve.  Per buffer
// b: s_full[b] (S ready), p_full[b] (P ready, four warp arrivals) and
// p_empty[b] (the PV that read P done).  The MMA warp waits for the P of
// the slots in order, so no barrier runs two phases ahead of its waiter:
// S(n + 3) is issued after the wait for P(n), which the warpgroup signals
// after its wait for S(n); P(n + 3) follows S(n + 3); and a warpgroup at slot
// n that waits for the PV of its previous tile's slot n - nh has seen S(n),
// issued after PV(n - nh - 3), while PV(n - nh + 3) waits for P(n).
template <int D, bool DEC>
__device__ void mma_issuer_rot(const AttnParams& p, uint8_t* smem, Ctl* ctl, int lane) {
    using C = Cfg<D, DEC>;
    constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, 128, 0, 0);  // Q K-major, K K-major
    constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, D, 0, 1);   // P (TMEM), V MN-major
    const uint32_t tbase = ctl->tmem_base;
    const uint64_t dQ = ptx::smem_desc(ptx::smem_u32(smem + C::kOffQ), 16, 1024, 2);
    const uint32_t hi = (uint32_t)(dQ >> 32);
    const uint32_t lQ = (uint32_t)dQ;
    const uint32_t lK = (uint32_t)ptx::smem_desc(ptx::smem_u32(smem + C::kOffK), 16, 1024, 2);
    const uint32_t lV = (uint32_t)ptx::smem_desc(ptx::smem_u32(smem + C::kOffV), C::kPanelBytes, 1024, 2);
    uint32_t kv_cnt = 0, q_cnt = 0, oc0 = 0, oc1 = 0, n_taken = 0;
    // S buffer of the next S slot; S buffer and P-ready phase of the next PV slot
    uint32_t bs = 0, bp = 0, php = 0;

    for (;;) {
        const int ii = take_item_w(p, ctl, n_taken, kErrTimeoutMma, lane);
        if (ii < 0) return;
        const Item it = p.items[ii];
        const int T = it.pad;  // KV tiles of this item
        if (it.kind != kPrefill) { kv_cnt += T; continue; }
        const Group g = p.groups[it.group];
        const int nh = g.pad;
        if (!wait_bar_w(p, ctl, &ctl->q_full, q_cnt & 1, kErrTimeoutMma)) return;
        ++q_cnt;
        int2 mt_prev = make_int2(0, 0);  // metadata of tile j-1, read when its S was issued
        for (int j = 0; j <= T; ++j) {
            const int jj = j - 1;
            const uint32_t kj = kv_cnt + j, kp = kv_cnt + jj;
            const int st = kj % C::kStages, stp = kp % C::kStages;
            const int nk = (mt_prev.y + 15) >> 4;
            int2 mt_cur = mt_prev;
            if (j >= 1 && !wait_bar_w(p, ctl, &ctl->v_full[stp], (kp / C::kStages) & 1, kErrTimeoutMma)) return;
            if (j < T && !wait_bar_w(p, ctl, &ctl->k_full[st], (kj / C::kStages) & 1, kErrTimeoutMma)) return;
            for (int k = 0; k < nh; ++k) {
                if (j >= 1) {
                    if (!wait_bar_w(p, ctl, &ctl->p_full[bp], php, kErrTimeoutMma)) return;
                    if (jj == 0 &&
                        !wait_bar_w(p, ctl, &ctl->o_empty[k], ((k ? oc1 : oc0) & 1) ^ 1, kErrTimeoutMma))
                        return;
                }
                ptx::tc_fence_after();
                // S_k = Q_k K^T for tile j, first
                if (j < T) {
                    if (k == 0) mt_cur = ctl->tmeta[kj & 7];
                    const uint32_t kl = lK + (uint32_t)((st * C::kTileBytes) >> 4);
                    const uint32_t ql = lQ + (uint32_t)((k * C::kTileBytes) >> 4);
                    const uint32_t ts = tbase + bs * 128;
                    ptx::tc_mma_ss_e<0>(ts, ql, kl, hi, kIdescS);
#pragma unroll
                    for (int ks = 1; ks < D / 16; ++ks) {
                        const uint32_t off = (uint32_t)(((ks >> 2) * C::kPanelBytes + (ks & 3) * 32) >> 4);
                        ptx::tc_mma_ss_e<1>(ts, ql + off, kl + off, hi, kIdescS);
                    }
                    ptx::tc_commit_e(&ctl->s_full[bs]);
                    bs = bs == 2 ? 0 : bs + 1;
                }
                // then O_k += P_k V for tile j-1
                if (j >= 1) {
                    const uint32_t vl = lV + (uint32_t)((stp * C::kTileBytes) >> 4);
                    const uint32_t to = tbase + C::kTmemO + k * D, tp = tbase + bp * 128;
                    if (nk == kTileKeys / 16) {
#pragma unroll
                        for (int ks = 0; ks < kTileKeys / 16; ++ks)
                            ptx::tc_mma_ts_e<1>(to, tp + ks * 8, vl + ks * 128, hi, kIdescPV);
                    } else {
                        for (int ks = 0; ks < nk; ++ks) ptx::tc_mma_ts_e<1>(to, tp + ks * 8, vl + ks * 128, hi, kIdescPV);
                    }
                    ptx::tc_commit_e(&ctl->p_empty[bp]);
                    if (bp == 2) {
                        bp = 0;
                        php ^= 1;
                    } else {
                        ++bp;
                    }
                }
            }
            if (j >= 1) {
                ptx::tc_commit_e(&ctl->v_empty[stp]);
                if (jj == T - 1) {
                    ptx::tc_commit_e(&ctl->o_full);
                    ++oc0;
                    if (nh == 2) ++oc1;
                }
            }
            if (j < T) {
                ptx::tc_commit_e(&ctl->k_empty[st]);
                if (j == T - 1) ptx::tc_commit_e(&ctl->q_empty);
            }
            mt_prev = mt_cur;
        }
        kv_cnt += T;
    }
}

// ----------------------------------------------------- output helpers --

// Four consecutive output elements starting at idx (idx a multiple of 4).
__device__ __forceinline__ void store_out4(const AttnParams& p, int64_t idx, float4 v) {
    if (p.out_fp32) {
        *reinterpret_cast<float4*>(static_cast<float*>(p.out) + idx) = v;
    } else {
        uint2 w;
        w.x = ptx::pack_bf16x2(v.x, v.y);
        w.y = ptx::pack_bf16x2(v.z, v.w);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + idx) = w;
    }
}

__device__ __forceinline__ void store_out(const AttnParams& p, int64_t idx, float v) {
    if (p.out_fp32) static_cast<float*>(p.out)[idx] = v;
    else static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
}

// ------------------------------------------------------ decode (compute) --

template <int D, bool DEC, bool kHalf>
__device__ bool decode_item(const AttnParams& p, uint8_t* smem, Ctl* ctl, int ii, const Item& it, const Group& g,
                            uint32_t& kv_cnt, uint32_t& cs, uint32_t& mg, int cw, int lane) {
    using C = Cfg<D, DEC>;
    constexpr int NT = D / 8;   // 8-column output tiles
    const int G = p.G;
    const int M = g.nrows * G;
    const int kvh = g.head;
    const int gr = lane >> 2, tq = lane & 3;

    const int prow0 = gr < M ? p.pos[g.row0 + gr / G] : -1;
    const int prow1 = gr + 8 < M ? p.pos[g.row0 + (gr + 8) / G] : -1;

    // Q fragments (rows = query row x head, zero past M).  The decode-only
    // kernel has the registers to hold all of them; the mixed kernel stages Q
    // in shared memory as [16][D] bf16 (16-byte chunks XOR-swizzled by row)
    // and reads fragments back with ldmatrix (the merge scratch is free until
    // the tiles are done).
    constexpr int KSR = DEC ? D / 16 : 1;
    uint32_t qa_r[KSR][4];
    uint8_t* qs = smem + C::kOffScr;
    if constexpr (DEC) {
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(p.q);
        auto qword = [&](int m, int dim) -> uint32_t {
            if (m >= M) return 0u;
            const int64_t row = g.row0 + m / G;
            const int64_t h = (int64_t)kvh * G + m % G;
            return qw[((row * p.Hq + h) * D + dim) >> 1];
        };
#pragma unroll
        for (int ks = 0; ks < KSR; ++ks) {
            qa_r[ks][0] = qword(gr, ks * 16 + 2 * tq);
            qa_r[ks][1] = qword(gr + 8, ks * 16 + 2 * tq);
            qa_r[ks][2] = qword(gr, ks * 16 + 8 + 2 * tq);
            qa_r[ks][3] = qword(gr + 8, ks * 16 + 8 + 2 * tq);
        }
    } else {
        // the scratch must have been read by the merge warp (previous item)
        if (mg > 0 && !wait_bar(p, ctl, &ctl->merge_empty, (mg - 1) & 1, kErrTimeoutCompute)) return false;
        const int tid = cw * 32 + lane;
        const uint4* qg = reinterpret_cast<const uint4*>(p.q);
        for (int e = tid; e < kDecRows * (D / 8); e += 128) {
            const int m = e / (D / 8), c = e % (D / 8);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (m < M) {
                const int64_t row = g.row0 + m / G;
                const int64_t h = (int64_t)kvh * G + m % G;
                v = qg[((row * p.Hq + h) * D) / 8 + c];
            }
            *reinterpret_cast<uint4*>(qs + m * (D * 2) + ((c ^ (m & 7)) << 4)) = v;
        }
        if (!compute_sync(p, ctl, 0, cs)) return false;
    }
    const uint32_t qsa = ptx::smem_u32(qs);
    const int qrow = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row this lane addresses

    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    // lrun: fp32 probability sums (lse); rrun: sums of the bf16 values the PV
    // MMAs consume, P and its residual (output normaliser)
    float mrun0 = -INFINITY, mrun1 = -INFINITY, lrun0 = 0.f, lrun1 = 0.f, rrun0 = 0.f, rrun1 = 0.f;
    float lqb0 = 0.f, lqb1 = 0.f;  // see the residual check below
    const int key0 = cw * 32;
    const int T = it.pad;

    // A group of at most 8 live rows (M <= 8: one decode row per sequence
    // with G <= 8, or G = 1 with up to 8 rows) leaves the MMA's rows 8..15 as
    // padding.  There ("half" tiles) the padding rows carry the bf16 residual
    // p - bf16(p) of rows 0..7 through the same PV MMAs, so every tile gets
    // the exact product at no MMA cost, the padding rows' exponentials are
    // skipped, and rows 8..15 of O are folded into rows 0..7 at the end.
    for (int t = 0; t < T; ++t) {
        const uint32_t k = kv_cnt + t;
        const int st = k % C::kStages;
        const uint32_t ph = (k / C::kStages) & 1;
        if (!wait_bar(p, ctl, &ctl->k_full[st], ph, kErrTimeoutCompute)) return false;
        if (!wait_bar(p, ctl, &ctl->v_full[st], ph, kErrTimeoutCompute)) return false;
        const int2 mt = ctl->tmeta[k & 7];
        const int kt0 = mt.x, n = mt.y;
        if (key0 < n) {
            const uint32_t kb = ptx::smem_u32(smem + C::kOffK + st * C::kTileBytes);
            const uint32_t vb = ptx::smem_u32(smem + C::kOffV + st * C::kTileBytes);
            float s[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
                uint32_t qa0[4], qa1[4];
                if constexpr (DEC) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        qa0[i] = qa_r[(2 * kk) % KSR][i];
                        qa1[i] = qa_r[(2 * kk + 1) % KSR][i];
                    }
                } else {
                    const int c0 = 4 * kk + (lane >> 4);  // chunk of k-step 2kk
                    ptx::ldmatrix_x4(qsa + qrow * (D * 2) + ((c0 ^ (qrow & 7)) << 4), qa0[0], qa0[1], qa0[2],
                                     qa0[3]);
                    const int c1 = c0 + 2;  // k-step 2kk+1
                    ptx::ldmatrix_x4(qsa + qrow * (D * 2) + ((c1 ^ (qrow & 7)) << 4), qa1[0], qa1[1], qa1[2],
                                     qa1[3]);
                }
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int key = key0 + nt * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ptx::ldmatrix_x4(kb + sw128_off<D>(key, kk * 4 + (lane >> 3)), b0, b1, b2, b3);
                    ptx::mma_bf16_16816(s[nt], qa0, b0, b1);
                    ptx::mma_bf16_16816(s[nt], qa1, b2, b3);
                }
            }
            // mask (key inside the tile, causal key <= row position), scale to log2 units
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                for (int e = 0; e < (kHalf ? 2 : 4); ++e) {
                    const int key = key0 + nt * 8 + 2 * tq + (e & 1);
                    const int prow = (e >> 1) ? prow1 : prow0;
                    const bool vis = key < n && kt0 + key <= prow;
                    const float x = vis ? s[nt][e] * p.scale_log2 : -INFINITY;
                    s[nt][e] = x;
                    if (e >> 1) mx1 = fmaxf(mx1, x); else mx0 = fmaxf(mx0, x);
                }
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            if constexpr (!kHalf) {
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            }
            const float mn0 = fmaxf(mrun0, mx0), mn1 = fmaxf(mrun1, mx1);
            const float use0 = mn0 == -INFINITY ? 0.f : mn0;
            const float use1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = ptx::ex2(mrun0 - use0), al1 = kHalf ? al0 : ptx::ex2(mrun1 - use1);
            mrun0 = mn0;
            float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                s[nt][0] = ptx::ex2(s[nt][0] - use0);
                s[nt][1] = ptx::ex2(s[nt][1] - use0);
                sum0 += s[nt][0] + s[nt][1];
                if constexpr (!kHalf) {
                    s[nt][2] = ptx::ex2(s[nt][2] - use1);
                    s[nt][3] = ptx::ex2(s[nt][3] - use1);
                    sum1 += s[nt][2] + s[nt][3];
                }
            }
            lrun0 = lrun0 * al0 + sum0;
            rrun0 *= al0;
            if constexpr (!kHalf) {
                mrun1 = mn1;
                lrun1 = lrun1 * al1 + sum1;
                rrun1 *= al1;
            }
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    o[i][0] *= al0; o[i][1] *= al0;
                    o[i][2] *= al1; o[i][3] *= al1;
                }
            }
            const bool tail = key0 + 32 > n;
            // O += P V over this warp's 32 keys (two 16-key MMA steps).  Where
            // a row's weight sits on few keys the bf16 rounding of P does not
            // average away, so the bf16 residual p - bf16(p) goes through the
            // MMA too: in half tiles as rows 8..15 of the same MMA, otherwise
            // as a second MMA.  In the decode-only launch every full tile
            // takes the second MMA (a decode tile has MMA time to spare).  In
            // the launch with prefill items, where extra MMAs slow the whole
            // kernel, a full tile takes it on a sequence's first 128 keys
            // (rows may see few keys in all) and wherever this tile's share
            // of the error variance, sum p^2 / l^2, exceeds 1/16 for a row
            // (as in prefill_item; l here is this warp's sum over its quarter
            // of every tile so far, at most the row's total, so the test errs
            // towards the second MMA).  Two instantiations keep the rare path
            // out of the common loop.
            bool resid = DEC || kt0 < kTileKeys;
            if constexpr (!kHalf) {
                // The running max is exact here, so p <= 1 and a row whose
                // sum has reached 16 cannot need the pass: lqb, a lower bound
                // of the row's sum over this warp's keys (rescaled with it,
                // refreshed only while below 16), spares the shuffles on most
                // tiles.
                lqb0 *= al0;
                lqb1 *= al1;
                if (!resid && __any_sync(0xffffffffu, lqb0 < 16.f || lqb1 < 16.f)) {
                    float lq0 = lrun0 + __shfl_xor_sync(0xffffffffu, lrun0, 1);
                    float lq1 = lrun1 + __shfl_xor_sync(0xffffffffu, lrun1, 1);
                    lq0 += __shfl_xor_sync(0xffffffffu, lq0, 2);
                    lq1 += __shfl_xor_sync(0xffffffffu, lq1, 2);
                    lqb0 = lq0;
                    lqb1 = lq1;
                    bool r0 = mx0 != -INFINITY && ptx::ex2(mx0 - use0) * 16.f > lq0;
                    bool r1 = mx1 != -INFINITY && ptx::ex2(mx1 - use1) * 16.f > lq1;
                    if (__any_sync(0xffffffffu, r0 || r1)) {
                        float q0 = 0.f, q1 = 0.f;
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt) {
                            q0 += s[nt][0] * s[nt][0] + s[nt][1] * s[nt][1];
                            q1 += s[nt][2] * s[nt][2] + s[nt][3] * s[nt][3];
                        }
                        q0 += __shfl_xor_sync(0xffffffffu, q0, 1);
                        q1 += __shfl_xor_sync(0xffffffffu, q1, 1);
                        q0 += __shfl_xor_sync(0xffffffffu, q0, 2);
                        q1 += __shfl_xor_sync(0xffffffffu, q1, 2);
                        r0 = r0 && q0 * 16.f > lq0 * lq0;
                        r1 = r1 && q1 * 16.f > lq1 * lq1;
                    }
                    resid = __any_sync(0xffffffffu, r0 || r1);
                }
            }
            // bf16 residual of the pair (x, y) given its bf16 pack w
            auto lo_of = [](float x, float y, uint32_t w) {
                return ptx::pack_bf16x2(x - __uint_as_float(w << 16), y - __uint_as_float(w & 0xffff0000u));
            };
            auto pv = [&](auto precise_tag) {
                constexpr bool kPrecise = decltype(precise_tag)::value && !kHalf;
#pragma unroll
                for (int kst = 0; kst < 2; ++kst) {
                    uint32_t a[4];
                    a[0] = ptx::pack_bf16x2(s[2 * kst][0], s[2 * kst][1]);
                    a[2] = ptx::pack_bf16x2(s[2 * kst + 1][0], s[2 * kst + 1][1]);
                    if constexpr (kHalf) {
                        a[1] = lo_of(s[2 * kst][0], s[2 * kst][1], a[0]);
                        a[3] = lo_of(s[2 * kst + 1][0], s[2 * kst + 1][1], a[2]);
                    } else {
                        a[1] = ptx::pack_bf16x2(s[2 * kst][2], s[2 * kst][3]);
                        a[3] = ptx::pack_bf16x2(s[2 * kst + 1][2], s[2 * kst + 1][3]);
                    }
                    const int kbase = key0 + kst * 16;
                    if (kbase >= n) break;
                    if constexpr (kHalf) {
                        rrun0 += (bf16x2_sum(a[0]) + bf16x2_sum(a[2])) + (bf16x2_sum(a[1]) + bf16x2_sum(a[3]));
                    } else {
                        rrun0 += bf16x2_sum(a[0]) + bf16x2_sum(a[2]);
                        rrun1 += bf16x2_sum(a[1]) + bf16x2_sum(a[3]);
                    }
                    uint32_t alo[4] = {0u, 0u, 0u, 0u};
                    if constexpr (kPrecise) {
                        alo[0] = lo_of(s[2 * kst][0], s[2 * kst][1], a[0]);
                        alo[1] = lo_of(s[2 * kst][2], s[2 * kst][3], a[1]);
                        alo[2] = lo_of(s[2 * kst + 1][0], s[2 * kst + 1][1], a[2]);
                        alo[3] = lo_of(s[2 * kst + 1][2], s[2 * kst + 1][3], a[3]);
                        rrun0 += bf16x2_sum(alo[0]) + bf16x2_sum(alo[2]);
                        rrun1 += bf16x2_sum(alo[1]) + bf16x2_sum(alo[3]);
                    }
                    // V rows past the valid keys may hold anything (even NaN): zero them
                    uint32_t m0 = 0xffffffffu, m1 = 0xffffffffu;
                    if (tail) {
                        const int k0 = kbase + 2 * tq;
                        m0 = (k0 < n ? 0x0000ffffu : 0u) | (k0 + 1 < n ? 0xffff0000u : 0u);
                        m1 = (k0 + 8 < n ? 0x0000ffffu : 0u) | (k0 + 9 < n ? 0xffff0000u : 0u);
                    }
                    const int vkey = kbase + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                    for (int dp = 0; dp < D / 16; ++dp) {
                        uint32_t b0, b1, b2, b3;
                        ptx::ldmatrix_x4_trans(vb + sw128_off<D>(vkey, dp * 2 + (lane >> 4)), b0, b1, b2, b3);
                        ptx::mma_bf16_16816(o[2 * dp], a, b0 & m0, b1 & m1);
                        ptx::mma_bf16_16816(o[2 * dp + 1], a, b2 & m0, b3 & m1);
                        if constexpr (kPrecise) {
                            ptx::mma_bf16_16816(o[2 * dp], alo, b0 & m0, b1 & m1);
                            ptx::mma_bf16_16816(o[2 * dp + 1], alo, b2 & m0, b3 & m1);
                        }
                    }
                }
            };
            if (kHalf || !resid) pv(std::false_type{});
            else pv(std::true_type{});
        }
        if (!compute_sync(p, ctl, 0, cs)) return false;
        if (cw == 0 && lane == 0) {
            ptx::mbar_arrive(&ctl->k_empty[st]);
            ptx::mbar_arrive(&ctl->v_empty[st]);
        }
    }
    if constexpr (kHalf) {
        // rows 8..15 hold (p - bf16(p)) V of rows 0..7
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            o[i][0] += o[i][2];
            o[i][1] += o[i][3];
            o[i][2] = o[i][3] = 0.f;
        }
    }
    kv_cnt += T;

    // combine the four warps' states (each saw a different quarter of every tile)
    lrun0 += __shfl_xor_sync(0xffffffffu, lrun0, 1);
    lrun0 += __shfl_xor_sync(0xffffffffu, lrun0, 2);
    lrun1 += __shfl_xor_sync(0xffffffffu, lrun1, 1);
    lrun1 += __shfl_xor_sync(0xffffffffu, lrun1, 2);
    rrun0 += __shfl_xor_sync(0xffffffffu, rrun0, 1);
    rrun0 += __shfl_xor_sync(0xffffffffu, rrun0, 2);
    rrun1 += __shfl_xor_sync(0xffffffffu, rrun1, 1);
    rrun1 += __shfl_xor_sync(0xffffffffu, rrun1, 2);
    // hand the four warps' states to the merge warp through the scratch
    if (DEC && mg > 0 && !wait_bar(p, ctl, &ctl->merge_empty, (mg - 1) & 1, kErrTimeoutCompute)) return false;
    float* scr = reinterpret_cast<float*>(smem + C::kOffScr);  // [4][16][D]
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        const int c = i * 8 + 2 * tq;
        *reinterpret_cast<float2*>(&scr[(cw * kDecRows + gr) * D + c]) = make_float2(o[i][0], o[i][1]);
        *reinterpret_cast<float2*>(&scr[(cw * kDecRows + gr + 8) * D + c]) = make_float2(o[i][2], o[i][3]);
    }
    if (tq == 0) {
        ctl->dec_m[cw][gr] = mrun0;
        ctl->dec_l[cw][gr] = lrun0;
        ctl->dec_m[cw][gr + 8] = mrun1;
        ctl->dec_l[cw][gr + 8] = lrun1;
        ctl->dec_lr[cw][gr] = rrun0;
        ctl->dec_lr[cw][gr + 8] = rrun1;
    }
    if (cw == 0 && lane == 0) ctl->merge_item = ii;
    ptx::mbar_arrive(&ctl->merge_full);
    ++mg;
    return true;
}

// Merge warp: for each decode item handed over by the compute warps, combine
// the four warps' (max, sums, unnormalised out) states of every query row
// and head (log-sum-exp), write the output, or, for one part of a split group,
// the normalised fp32 partial and its lse; then the last part to arrive
// (atomic counter after a fence) merges the group's parts and resets the
// counter.  Runs while the compute warps process the next item.
template <int D, bool DEC>
__device__ void merge_warp(const AttnParams& p, uint8_t* smem, Ctl* ctl, int lane) {
    using C = Cfg<D, DEC>;
    const float* scr = reinterpret_cast<const float*>(smem + C::kOffScr);  // [4][16][D]
    const int G = p.G;
    for (uint32_t n = 0;; ++n) {
        // The wait for the next hand-over spans whatever prefill work the
        // compute warps do in between, so it may take up to 30 wait limits;
        // it ends at once when another role aborts.
        bool ok = false;
        for (int r = 0; r < 30; ++r) {
            ok = __all_sync(0xffffffffu,
                            ptx::mbar_wait_sleep(&ctl->merge_full, n & 1, &ctl->abort, p.limit_ns, 1000));
            if (ok || *reinterpret_cast<volatile int*>(&ctl->abort)) break;
        }
        if (!ok) {
            fail(p, ctl, kErrTimeoutCompute);
            return;
        }
        const int ii = ctl->merge_item;
        if (ii < 0) return;
        const Item it = p.items[ii];
        const Group g = p.groups[it.group];
        const int M = g.nrows * G;  // rows m = query row x head, <= 16
        const int kvh = g.head;
        const bool split = g.n_parts > 1;
        // Lane m < M owns row m: the log-sum-exp weights of the four warps'
        // states, normalised by the bf16-probability sum the PV MMAs used.
        float fw[4] = {0.f, 0.f, 0.f, 0.f};
        float lse_row = -INFINITY;
        if (lane < M) {
            float mm = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w) mm = fmaxf(mm, ctl->dec_m[w][lane]);
            if (mm != -INFINITY) {
                float L = 0.f, LR = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    fw[w] = ptx::ex2(ctl->dec_m[w][lane] - mm);
                    L += ctl->dec_l[w][lane] * fw[w];
                    LR += ctl->dec_lr[w][lane] * fw[w];
                }
                const float inv = 1.f / LR;
#pragma unroll
                for (int w = 0; w < 4; ++w) fw[w] *= inv;
                lse_row = mm + log2f(L);
            }
        }
        float* part = split ? p.dec_part + (int64_t)(g.slot + it.part) * kDecRows * D : nullptr;
        // elements as float4 chunks of D/4 per row; kIt uniform trips per lane
        const int n_chunks = M * (D / 4);
        const int kIt = (n_chunks + 31) / 32;
        for (int k = 0; k < kIt; ++k) {
            const int c = k * 32 + lane;
            const int m = min(c / (D / 4), M - 1), d = (c % (D / 4)) * 4;
            float f[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) f[w] = __shfl_sync(0xffffffffu, fw[w], m);
            if (c < n_chunks) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float4 v = *reinterpret_cast<const float4*>(&scr[(w * kDecRows + m) * D + d]);
                    acc.x += f[w] * v.x; acc.y += f[w] * v.y; acc.z += f[w] * v.z; acc.w += f[w] * v.w;
                }
                if (split) {
                    *reinterpret_cast<float4*>(part + m * D + d) = acc;
                } else {
                    const int64_t row = g.row0 + m / G;
                    const int64_t h = (int64_t)kvh * G + m % G;
                    store_out4(p, (row * p.Hq + h) * D + d, acc);
                }
            }
        }
        if (lane < M) {
            if (split) {
                p.dec_lse[(int64_t)(g.slot + it.part) * kDecRows + lane] = lse_row;
            } else if (p.lse) {
                const int64_t row = g.row0 + lane / G;
                p.lse[row * p.Hq + (int64_t)kvh * G + lane % G] = lse_row * kLn2;
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ctl->merge_empty);  // scratch free for the next item
        if (!split) continue;
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&p.counters[2 * it.group], 1) == g.n_parts - 1;
        if (!__shfl_sync(0xffffffffu, last, 0)) continue;
        __threadfence();
        // last part: merge the group's parts by log-sum-exp (lane m owns row m)
        const float* base = p.dec_part + (int64_t)g.slot * kDecRows * D;
        const float* lbase = p.dec_lse + (int64_t)g.slot * kDecRows;
        const int np = g.n_parts;
        float mm = -INFINITY, invL = 0.f;
        if (lane < M) {
            for (int q = 0; q < np; ++q) mm = fmaxf(mm, __ldcg(lbase + q * kDecRows + lane));
            if (mm != -INFINITY) {
                float L = 0.f;
                for (int q = 0; q < np; ++q) L += ptx::ex2(__ldcg(lbase + q * kDecRows + lane) - mm);
                invL = 1.f / L;
                lse_row = mm + log2f(L);
            } else {
                lse_row = -INFINITY;
            }
        }
        for (int k = 0; k < kIt; ++k) {
            const int c = k * 32 + lane;
            const int m = min(c / (D / 4), M - 1), d = (c % (D / 4)) * 4;
            const float mm_m = __shfl_sync(0xffffffffu, mm, m);
            const float inv_m = __shfl_sync(0xffffffffu, invL, m);
            if (c < n_chunks) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                if (mm_m != -INFINITY) {
                    int q = 0;
                    for (; q + 2 <= np; q += 2) {  // two parts per step: independent loads in flight
                        const float l0 = __ldcg(lbase + q * kDecRows + m);
                        const float l1 = __ldcg(lbase + (q + 1) * kDecRows + m);
                        const float4 v0 = __ldcg(reinterpret_cast<const float4*>(base + ((int64_t)q * kDecRows + m) * D + d));
                        const float4 v1 =
                            __ldcg(reinterpret_cast<const float4*>(base + ((int64_t)(q + 1) * kDecRows + m) * D + d));
                        const float w0 = ptx::ex2(l0 - mm_m) * inv_m, w1 = ptx::ex2(l1 - mm_m) * inv_m;
                        acc.x += w0 * v0.x + w1 * v1.x;
                        acc.y += w0 * v0.y + w1 * v1.y;
                        acc.z += w0 * v0.z + w1 * v1.z;
                        acc.w += w0 * v0.w + w1 * v1.w;
                    }
                    if (q < np) {
                        const float l0 = __ldcg(lbase + q * kDecRows + m);
                        const float4 v0 = __ldcg(reinterpret_cast<const float4*>(base + ((int64_t)q * kDecRows + m) * D + d));
                        const float w0 = ptx::ex2(l0 - mm_m) * inv_m;
                        acc.x += w0 * v0.x; acc.y += w0 * v0.y; acc.z += w0 * v0.z; acc.w += w0 * v0.w;
                    }
                }
                const int64_t row = g.row0 + m / G;
                const int64_t h = (int64_t)kvh * G + m % G;
                store_out4(p, (row * p.Hq + h) * D + d, acc);
            }
        }
        if (lane < M && p.lse) {
            const int64_t row = g.row0 + lane / G;
            p.lse[row * p.Hq + (int64_t)kvh * G + lane % G] = lse_row * kLn2;
        }
        __syncwarp();
        if (lane == 0) p.counters[2 * it.group] = 0;  // ready for the next launch
    }
}

// ----------------------------------------------------- prefill (compute) --

// The careful instance of a tile's exponentials, out of line so that the
// common loop's code stays as it is: S is read back from TMEM 16 columns at a
// time, P and its bf16 residual are written over the same columns (P of keys
// 16ks.. in columns 16ks..16ks+7, the residual in 16ks+8..16ks+15), then one
// 128-column read moves them to where the PV passes take them: P pairs in
// columns 0..63, residual pairs in 64..127.  Returns (sum p, sum p^2).
__device__ __noinline__ float2 careful_exps(uint32_t tS, int lim, float sl, float nm) {
    float sum = 0.f, sq = 0.f;
#pragma unroll 1
    for (int ks = 0; ks < 8; ++ks) {
        float v[16];
        ptx::tmem_ld16(tS + 16 * ks, v);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int col = 16 * ks + 2 * i;
            const float a = col < lim ? ptx::ex2(fmaf(v[2 * i], sl, nm)) : 0.f;
            const float b = col + 1 < lim ? ptx::ex2(fmaf(v[2 * i + 1], sl, nm)) : 0.f;
            sum += a + b;
            sq = fmaf(a, a, fmaf(b, b, sq));
            pk[i] = ptx::pack_bf16x2(a, b);
            pk[8 + i] = ptx::pack_bf16x2(a - __uint_as_float(pk[i] << 16), b - __uint_as_float(pk[i] & 0xffff0000u));
        }
        ptx::tmem_st16(tS + 16 * ks, pk);
    }
    ptx::tmem_wait_st();
    float r[128];
    ptx::tmem_ld128(tS, r);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(r);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        ptx::tmem_st8(tS + 8 * ks, w + 16 * ks);
        ptx::tmem_st8(tS + 64 + 8 * ks, w + 16 * ks + 8);
    }
    return make_float2(sum, sq);
}

// Second PV pass of one softmax warp (quarter q of warpgroup k) for the tile
// in V stage st: O_k += R V over this warp's 32 rows, R = p - bf16(p) in
// TMEM columns 64..127 of the tile's S buffer sbuf (keys 2i, 2i+1 in column
// 64 + i), every other row masked out of the MMA.  The warp issues it
// itself, so the MMA warp's loop is the same whether or not a tile needs
// it, and its completion is this warp's P-ready arrival (tcgen05.commit onto
// p_full): the MMA warp's own pass over O_k for this tile starts only after
// it.  The pass before has completed already: with two S buffers the S MMA
// of this tile, whose completion this warp waited for, was issued after it;
// with three the caller waits for it.  O_k is zero before an item's first
// tile.
template <int D, bool DEC>
__device__ bool residual_pass(const AttnParams& p, uint8_t* smem, Ctl* ctl, int k, int q, int lane, int st,
                              uint32_t ph, int n, uint32_t sbuf) {
    using C = Cfg<D, DEC>;
    constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, D, 0, 1);  // as the MMA warp's PV
    if (!wait_bar(p, ctl, &ctl->v_full[st], ph, kErrTimeoutCompute)) return false;
    if (n & (kBlock - 1)) {
        // V rows past the valid keys may hold anything (NaN times a zero
        // residual is NaN): zero them, as warpgroup 0 also does before its PV
        uint8_t* vs = smem + C::kOffV + st * C::kTileBytes;
        const int nz = ((n + 15) & ~15) - n;
        for (int c = lane; c < nz * (D / 8); c += 32) {
            const int r = n + c / (D / 8), cc = c % (D / 8);
            *reinterpret_cast<uint4*>(vs + (cc >> 3) * C::kPanelBytes + r * 128 + (cc & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        ptx::fence_proxy_async_smem();
    }
    __syncwarp();
    ptx::tc_fence_after();
    const uint64_t dV = ptx::smem_desc(ptx::smem_u32(smem + C::kOffV), C::kPanelBytes, 1024, 2);
    const uint32_t hi = (uint32_t)(dV >> 32);
    const uint32_t vl = (uint32_t)dV + (uint32_t)((st * C::kTileBytes) >> 4);
    const uint32_t to = ctl->tmem_base + C::kTmemO + k * D, ta = ctl->tmem_base + sbuf * 128 + 64;
    const uint32_t m0 = q == 0 ? 0u : ~0u, m1 = q == 1 ? 0u : ~0u, m2 = q == 2 ? 0u : ~0u, m3 = q == 3 ? 0u : ~0u;
    const int nk = (n + 15) >> 4;
    for (int ks = 0; ks < nk; ++ks) ptx::tc_mma_ts_masked_e(to, ta + ks * 8, vl + ks * 128, hi, kIdescPV, m0, m1, m2, m3);
    ptx::tc_commit_e(&ctl->p_full[sbuf]);
    return true;
}

template <int D, bool DEC>
__device__ bool prefill_item(const AttnParams& p, uint8_t* smem, Ctl* ctl, const Item& it, const Group& g,
                             uint32_t& kv_cnt, uint32_t& sk, uint32_t& pvk, uint32_t& ok_cnt, uint32_t& cs, int k,
                             int r0, int qrows, int head, int warp, int lane) {
    using C = Cfg<D, DEC>;
    const int quarter = warp & 3;
    const int ri = quarter * 32 + lane;  // tile row = TMEM lane
    // r0 / qrows / head: first row, rows and query head of query tile k
    // (computed by the caller)
    const bool valid = ri < qrows;
    const int prow = valid ? p.pos[r0 + ri] : -1;
    const uint32_t tlane = ctl->tmem_base + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tO = tlane + C::kTmemO + k * D;  // O_k
    const int T = it.pad;
    const int nh = g.pad;
    // rotating S buffers: sk counts the slots of every earlier prefill item
    const uint32_t sb = sk;
    if constexpr (C::kRot) sk += (uint32_t)(T * nh);
    const float sl = p.scale_log2;
    // l: sum of the fp32 probabilities: the normaliser of the output and the
    // lse.  P reaches the PV MMA rounded to bf16.  lg_l = log2(l).
    float m = -INFINITY, l = 0.f, lg_l = -INFINITY;

    for (int j = 0; j < T; ++j) {
        const uint32_t kj = kv_cnt + j;
        const int st = kj % C::kStages;
        const uint32_t ph = (kj / C::kStages) & 1;
        // this tile's S buffer and phase; the S buffer of this query tile's
        // previous tile (whose PV is the last write into O_k before this
        // tile's) and the phase of its PV-done barrier
        uint32_t sbuf, sph, pb, pph;
        if constexpr (C::kRot) {
            const uint32_t n = sb + (uint32_t)(j * nh + k), np = n - (uint32_t)nh;
            sbuf = n % 3;
            sph = (n / 3) & 1;
            pb = np % 3;
            pph = (np / 3) & 1;
        } else {
            sbuf = k;
            sph = sk & 1;
            ++sk;
            pb = k;
            pph = (pvk - 1) & 1;
        }
        const uint32_t tS = tlane + sbuf * 128;  // S, later P (cols 0..63) and its residual (64..127)
        if (!wait_bar(p, ctl, &ctl->s_full[sbuf], sph, kErrTimeoutCompute)) return false;
        if (!wait_bar(p, ctl, &ctl->meta_full[kj & 7], (kj >> 3) & 1, kErrTimeoutCompute)) return false;
        ptx::tc_fence_after();
        const int2 mt = ctl->tmeta[kj & 7];
        const int kt0 = mt.x, n = mt.y;
        const int lim = max(0, min(n, prow - kt0 + 1));  // visible columns of this row
        float s[128];
        ptx::tmem_ld128(tS, s);
        if (!__all_sync(0xffffffffu, lim >= kTileKeys)) {
            // some row of the warp does not see the whole tile: mask in place
            // (a select, so garbage past the valid keys cannot leak through)
#pragma unroll
            for (int c = 0; c < 128; ++c) s[c] = c < lim ? s[c] : -INFINITY;
        }
        float mx;
        {
            // row max: four independent chains of 3-input max, then a tree
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 128; c += 8) {
                m4[0] = ptx::fmax3(m4[0], s[c], s[c + 1]);
                m4[1] = ptx::fmax3(m4[1], s[c + 2], s[c + 3]);
                m4[2] = ptx::fmax3(m4[2], s[c + 4], s[c + 5]);
                m4[3] = ptx::fmax3(m4[3], s[c + 6], s[c + 7]);
            }
            mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        float alpha = 1.f;
        bool resc = false, careful = false;
        if (lim > 0) {
            const float ms = mx * sl;
            // Residual check, before m moves (see below): a tile can need the
            // second PV pass only if its largest p exceeds l_old / 4, i.e.
            // ms + 2 > m + log2(l_old) in log2 units (always on a row's first
            // tile, where l_old = 0).
            careful = ms + 2.f > m + lg_l;
            // keep the running max unless the new one is larger by more than
            // 8 (log2 units): values stay <= 256, rescales of O become rare
            if (ms > m + 8.f) {
                alpha = ptx::ex2(m - ms);
                resc = j > 0;
                m = ms;
            }
        }
        // one warp vote for both (a second only when one of them is set)
        uint32_t vote = 0u;
        if (__any_sync(0xffffffffu, resc || careful))
            vote = (__any_sync(0xffffffffu, resc) ? 1u : 0u) | (__any_sync(0xffffffffu, careful) ? 2u : 0u);
        if (vote & 1u) {
            // O_k must hold PV_k(j-1) before it is scaled
            if (!wait_bar(p, ctl, &ctl->p_empty[pb], pph, kErrTimeoutCompute)) return false;
            ptx::tc_fence_after();
            const float f = resc ? alpha : 1.f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                float ov[32];
                ptx::tmem_ld32(tO + c * 32, ov);
#pragma unroll
                for (int i = 0; i < 32; ++i) ov[i] *= f;
                ptx::tmem_st32(tO + c * 32, ov);
            }
            ptx::tmem_wait_st();
        }
        // Probabilities p = 2^(s*scale*log2e - m) on f32x2 pairs (masked
        // scores are -inf and give 0), summed in two packed accumulators; P
        // goes to TMEM as bf16 pairs, keys 2i and 2i+1 in column i (columns
        // 0..63), for the MMA warp's PV pass.
        //
        // The bf16 rounding of p (relative error up to 2^-8) averages away
        // over many keys of similar weight, but not where a row's weight sits
        // on a few keys.  The PV error this tile adds to a row has a variance
        // proportional to sum_j p_j^2 / l^2 (l: every probability so far, so
        // that share only falls as later tiles add mass).  Where it exceeds
        // 1/16 this warp sends the residual p - bf16(p) (columns 64..127)
        // through a second PV pass of its own, which leaves the product with
        // p to about 2^-16.  The residual and the squares cost instructions,
        // so a second, careful instance of the loop computes them; it is
        // taken only where the bound sum p^2 / (l_old + sum)^2 <= max p /
        // (4 l_old) cannot rule the pass out.
        const uint64_t sl2 = ptx::f2pack(sl, sl);
        const float nm = m == -INFINITY ? 0.f : -m;
        const uint64_t nm2 = ptx::f2pack(nm, nm);
        uint64_t acc2[2] = {0ull, 0ull};
        float sum, sumsq = 0.f;
        if (vote & 2u) {
            const float2 r = careful_exps(tS, lim, sl, nm);
            sum = r.x;
            sumsq = r.y;
        } else {
            // two stores of 32 columns (64 keys each): against one store per
            // 16 keys, +1.8 % at D = 64 and +0.3 to +0.7 % at D = 128
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int col = 64 * ks + 2 * i;
                    float a, b;
                    ptx::f2unpack(ptx::ffma2(ptx::f2pack(s[col], s[col + 1]), sl2, nm2), a, b);
                    a = ptx::ex2(a);
                    b = ptx::ex2(b);
                    acc2[i & 1] = ptx::fadd2(acc2[i & 1], ptx::f2pack(a, b));
                    pk[i] = ptx::pack_bf16x2(a, b);
                }
                ptx::tmem_st32(tS + 32 * ks, reinterpret_cast<const float*>(pk));
            }
            float a0, a1, b0, b1;
            ptx::f2unpack(acc2[0], a0, a1);
            ptx::f2unpack(acc2[1], b0, b1);
            sum = (a0 + a1) + (b0 + b1);
        }
        l = l * alpha + sum;
        lg_l = ptx::lg2(l);  // for the next tile's check (off this tile's chain)
        const bool wresid = (vote & 2u) && __any_sync(0xffffffffu, sumsq * 16.f > l * l);
        if (k == 0 && (n & (kBlock - 1))) {
            // The tile ends inside a block: rows [n, ceil16(n)) of the V stage
            // may be pool rows past L_s holding anything.  The PV MMA covers
            // whole 16-row steps, so zero them (P is 0 there).  Warpgroup 0's
            // PV comes first, so this also covers warpgroup 1.
            if (!wait_bar(p, ctl, &ctl->v_full[st], ph, kErrTimeoutCompute)) return false;
            const int nz = ((n + 15) & ~15) - n;
            uint8_t* vs = smem + C::kOffV + st * C::kTileBytes;
            const int chunks = nz * (D / 8);
            for (int c = ri; c < chunks; c += 128) {
                const int r = n + c / (D / 8), cc = c % (D / 8);
                *reinterpret_cast<uint4*>(vs + (cc >> 3) * C::kPanelBytes + r * 128 + (cc & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
            }
            ptx::fence_proxy_async_smem();
        }
        // P ready: one arrival per warp (p_full counts the four warps), made
        // by lane 0 once the warp's TMEM stores are done, or by the
        // completion of the warp's residual pass
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (wresid) {
            if constexpr (C::kRot) {
                // with rotating buffers this tile's S can complete before the
                // PV of the previous tile into O_k is issued: wait for it
                if (j > 0 && !wait_bar(p, ctl, &ctl->p_empty[pb], pph, kErrTimeoutCompute)) return false;
            }
            if (!residual_pass<D, DEC>(p, smem, ctl, k, quarter, lane, st, ph, n, sbuf)) return false;
        } else if (lane == 0) {
            ptx::mbar_arrive(&ctl->p_full[sbuf]);
        }
        ++pvk;
    }
    kv_cnt += T;

    // epilogue: O_k row in 32-column chunks
    if (!wait_bar(p, ctl, &ctl->o_full, ok_cnt & 1, kErrTimeoutCompute)) return false;
    ++ok_cnt;
    ptx::tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse2 = l > 0.f ? m + log2f(l) : -INFINITY;
    const bool split = g.n_parts > 1;
    const int64_t slot0 = split ? ((int64_t)(g.slot + it.part) * 2 + k) * kTileRows : 0;
    const int64_t obase = ((int64_t)(r0 + ri) * p.Hq + head) * D;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
        float ov[32];
        ptx::tmem_ld32(tO + c * 32, ov);
        {
            // O_k starts the next item at zero (every PV MMA accumulates)
            float z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0.f;
            ptx::tmem_st32(tO + c * 32, z);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) ov[i] *= inv;
        if (split) {
            float4* dst = reinterpret_cast<float4*>(p.pre_part + (slot0 + ri) * D + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
        } else if (valid) {
            if (p.out_fp32) {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + obase + c * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i) dst[i] = make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
            } else {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + obase + c * 32);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint4 w;
                    w.x = ptx::pack_bf16x2(ov[8 * i], ov[8 * i + 1]);
                    w.y = ptx::pack_bf16x2(ov[8 * i + 2], ov[8 * i + 3]);
                    w.z = ptx::pack_bf16x2(ov[8 * i + 4], ov[8 * i + 5]);
                    w.w = ptx::pack_bf16x2(ov[8 * i + 6], ov[8 * i + 7]);
                    dst[i] = w;
                }
            }
        }
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    ptx::mbar_arrive(&ctl->o_empty[k]);
    if (!split) {
        if (valid && p.lse) p.lse[(int64_t)(r0 + ri) * p.Hq + head] = lse2 * kLn2;
        return true;
    }
    // split group: this part is written; the last part to arrive merges
    p.pre_lse[slot0 + ri] = lse2;
    __threadfence();
    if (!compute_sync(p, ctl, k, cs)) return false;
    if (ri == 0) {
        const int old = atomicAdd(&p.counters[2 * it.group + k], 1);
        ctl->flag_last[k] = (old == g.n_parts - 1);
    }
    if (!compute_sync(p, ctl, k, cs)) return false;
    if (ctl->flag_last[k]) {
        __threadfence();
        if (valid) {
            float mm = -INFINITY;
            for (int q = 0; q < g.n_parts; ++q)
                mm = fmaxf(mm, __ldcg(p.pre_lse + ((int64_t)(g.slot + q) * 2 + k) * kTileRows + ri));
            float L = 0.f;
            if (mm != -INFINITY)
                for (int q = 0; q < g.n_parts; ++q)
                    L += ptx::ex2(__ldcg(p.pre_lse + ((int64_t)(g.slot + q) * 2 + k) * kTileRows + ri) - mm);
            const float invL = L > 0.f ? 1.f / L : 0.f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                float acc[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[i] = 0.f;
                if (mm != -INFINITY) {
                    for (int q = 0; q < g.n_parts; ++q) {
                        const int64_t sq = ((int64_t)(g.slot + q) * 2 + k) * kTileRows + ri;
                        const float f = ptx::ex2(__ldcg(p.pre_lse + sq) - mm) * invL;
                        const float4* src = reinterpret_cast<const float4*>(p.pre_part + sq * D + c * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4 v = __ldcg(src + i);
                            acc[4 * i] += f * v.x; acc[4 * i + 1] += f * v.y;
                            acc[4 * i + 2] += f * v.z; acc[4 * i + 3] += f * v.w;
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) store_out(p, obase + c * 32 + i, acc[i]);
            }
            if (p.lse) p.lse[(int64_t)(r0 + ri) * p.Hq + head] = L > 0.f ? (mm + log2f(L)) * kLn2 : -INFINITY;
        }
        if (ri == 0) p.counters[2 * it.group + k] = 0;  // ready for the next launch
    }
    return compute_sync(p, ctl, k, cs);
}

template <int D, bool DEC>
__device__ void compute(const AttnParams& p, uint8_t* smem, Ctl* ctl, int warp, int lane) {
    using C = Cfg<D, DEC>;
    const int wg = (warp - C::kFirstCompute) >> 2;  // softmax warpgroup 0 or 1
    const int cw = (warp - C::kFirstCompute) & 3;
    uint32_t kv_cnt = 0, sk = 0, pvk = 0, ok_cnt = 0, cs = 0, n_taken = 0, mg = 0;
    if constexpr (!DEC) {
        if (p.has_prefill) {
            // O_wg starts at zero; every PV MMA accumulates (the epilogue
            // clears it again for the next item).  The MMA warp first writes
            // it after this warpgroup's first P-ready signal.
            const uint32_t tO = ctl->tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + C::kTmemO + wg * D;
            float z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) ptx::tmem_st32(tO + c * 32, z);
            ptx::tmem_wait_st();
        }
    }
    for (;;) {
        const int ii = take_item(p, ctl, n_taken, kErrTimeoutCompute);
        if (ii < 0) {
            if (wg == 0) {  // tell the merge warp there is nothing more
                if (mg > 0 && !wait_bar(p, ctl, &ctl->merge_empty, (mg - 1) & 1, kErrTimeoutCompute)) return;
                if (cw == 0 && lane == 0) ctl->merge_item = -1;
                ptx::mbar_arrive(&ctl->merge_full);
            }
            return;
        }
        const Item it = p.items[ii];
        const Group g = p.groups[it.group];
        bool ok = true;
        if (DEC || it.kind == kDecode) {
            // decode items run on warpgroup 0; warpgroup 1 only keeps count
            if (wg == 0) {
                // half tiles for groups of at most 8 live rows (the bf16
                // residual of P rides in rows 8..15 of the same MMAs)
                if (g.nrows * p.G <= 8)
                    ok = decode_item<D, DEC, true>(p, smem, ctl, ii, it, g, kv_cnt, cs, mg, cw, lane);
                else
                    ok = decode_item<D, DEC, false>(p, smem, ctl, ii, it, g, kv_cnt, cs, mg, cw, lane);
            }
            else kv_cnt += it.pad;
        } else if constexpr (!DEC) {
            if (wg < g.pad) {
                ok = prefill_item<D, DEC>(p, smem, ctl, it, g, kv_cnt, sk, pvk, ok_cnt, cs, wg, qtile_row0(p, g, wg),
                                          qtile_rows(p, g, wg), qtile_head(p, g, wg), warp, lane);
            } else {  // a one-head item: only the o_full phase and the ring positions move on
                kv_cnt += it.pad;
                if constexpr (Cfg<D, DEC>::kRot) {
                    // The S buffers' barriers move on with this item's slots,
                    // which are all warpgroup 0's: wait until the item is done,
                    // so that this warpgroup's next wait on a buffer is at most
                    // one phase ahead of it (a parity wait cannot tell further)
                    sk += (uint32_t)it.pad;
                    ok = wait_bar(p, ctl, &ctl->o_full, ok_cnt & 1, kErrTimeoutCompute);
                }
                ++ok_cnt;
            }
        }
        if (!ok) return;
    }
}

template <int D, bool DEC>
__global__ void __launch_bounds__(Cfg<D, DEC>::kThreads, 1)
    msa_attention_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmK64, const __grid_constant__ CUtensorMap tmK32,
                         const __grid_constant__ CUtensorMap tmK16, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmV64, const __grid_constant__ CUtensorMap tmV32,
                         const __grid_constant__ CUtensorMap tmV16, const __grid_constant__ CUtensorMap tmQ) {
    using C = Cfg<D, DEC>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + C::kOffCtl);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Decode-only launches are programmatic dependents of the kernel before
    // them (normally the append of the step's K/V rows): the set-up below
    // (barriers, tensor-map prefetch) overlaps that kernel, and nothing in
    // global memory is touched before pdl_wait (a no-op in a launch without
    // the attribute).  This grid does not trigger its own dependents early:
    // the next kernel then launches as it completes (an early trigger let
    // the next append's CTAs sit beside these and cost 3 % per step).

    if (threadIdx.x == 0) {
        for (int s = 0; s < 8; ++s) {
            ptx::mbar_init(&ctl->k_full[s], 1);
            ptx::mbar_init(&ctl->k_empty[s], 1);
            ptx::mbar_init(&ctl->v_full[s], 1);
            ptx::mbar_init(&ctl->v_empty[s], 1);
        }
        ptx::mbar_init(&ctl->q_full, 1);
        ptx::mbar_init(&ctl->q_empty, 1);
        for (int b = 0; b < 3; ++b) {
            ptx::mbar_init(&ctl->s_full[b], 1);
            ptx::mbar_init(&ctl->p_full[b], 4);  // one arrival per softmax warp
            ptx::mbar_init(&ctl->p_empty[b], 1);
        }
        for (int k = 0; k < 2; ++k) {
            ptx::mbar_init(&ctl->o_empty[k], 128);
            ptx::mbar_init(&ctl->csync[k], 128);
        }
        ptx::mbar_init(&ctl->o_full, 1);
        ptx::mbar_init(&ctl->drain, 1);
        ptx::mbar_init(&ctl->merge_full, 128);
        ptx::mbar_init(&ctl->merge_empty, 1);
        for (int r = 0; r < 4; ++r) {
            ptx::mbar_init(&ctl->item_full[r], 1);
            // consumers of every item id: the compute threads, the MMA thread, the V producer
            ptx::mbar_init(&ctl->item_empty[r], C::kComputeWarps * 32 + (DEC ? 0 : 1) + 1);
        }
        for (int r = 0; r < 8; ++r) ptx::mbar_init(&ctl->meta_full[r], 1);
        ctl->abort = 0;
        ctl->flag_last[0] = ctl->flag_last[1] = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmK64);
        ptx::prefetch_tmap(&tmK32);
        ptx::prefetch_tmap(&tmK16);
        ptx::prefetch_tmap(&tmV);
        ptx::prefetch_tmap(&tmV64);
        ptx::prefetch_tmap(&tmV32);
        ptx::prefetch_tmap(&tmV16);
        if (!DEC) ptx::prefetch_tmap(&tmQ);
    }
    if (!DEC && warp == 1 && p.has_prefill) {
        ptx::tmem_alloc(&ctl->tmem_base, C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::pdl_wait();
    // Each role sits inside the branch that sets its register budget.
    if (warp < C::kFirstCompute) {
        if constexpr (!DEC) ptx::setmaxnreg_dec<C::kRegsLow>();
        if (warp == 0) {
            if (lane == 0) producer<D, DEC, true>(p, smem, ctl, &tmK, &tmK64, &tmK32, &tmK16, &tmQ);
        } else if (warp == C::kVWarp) {
            if (lane == 0) producer<D, DEC, false>(p, smem, ctl, &tmV, &tmV64, &tmV32, &tmV16, &tmQ);
        } else if (warp == 1) {
            if constexpr (!DEC) {
                if (p.has_prefill) {
                    if constexpr (C::kRot)
                        mma_issuer_rot<D, DEC>(p, smem, ctl, lane);
                    else
                        mma_issuer<D, DEC>(p, smem, ctl, lane);
                    __syncwarp();
                    if (lane == 0) {
                        // every MMA lane 0 issued must have completed before TMEM is released
                        ptx::tc_commit(&ctl->drain);
                        static __shared__ int never;
                        never = 0;
                        ptx::mbar_wait(&ctl->drain, 0, &never, 100000000ull);
                    }
                }
            }
        } else if (warp == C::kMergeWarp) {
            merge_warp<D, DEC>(p, smem, ctl, lane);
        }
    } else if (DEC && warp == C::kMergeWarp) {
        merge_warp<D, DEC>(p, smem, ctl, lane);
    } else {
        if constexpr (!DEC) ptx::setmaxnreg_inc<C::kRegsHigh>();
        compute<D, DEC>(p, smem, ctl, warp, lane);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (!DEC && warp == 1 && p.has_prefill) ptx::tmem_dealloc(ctl->tmem_base, C::kTmemCols);
    if (threadIdx.x == 0) {
        // every CTA has stopped taking items once its producer saw the end of
        // the queue; the last CTA to finish leaves the queue reset for the
        // next launch with this workspace
        __threadfence();
        if (atomicAdd(&p.sched[1], 1) == (int)gridDim.x - 1) {
            p.sched[0] = 0;
            p.sched[1] = 0;
            __threadfence();
        }
    }
}

// ------------------------------------------------------------ host side --

// 3-D bf16 tensor map over [rows, heads, D] with a box of 64 x 1 x box_rows
// (tensor_maps.cpp: encoded once per thread and inputs).
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int D, int box_rows);

// Launch attributes of one kernel instantiation on the current device (a
// function attribute belongs to the device it was set on): done once per
// device, bit d of `done` marking device d.
template <int D, bool DEC>
static int configure_current_device() {
    using C = Cfg<D, DEC>;
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MSA_ERR_CUDA;
    const uint64_t bit = uint64_t(1) << dev;
    if (done.load(std::memory_order_acquire) & bit) return MSA_OK;
    if (cudaFuncSetAttribute(msa_attention_kernel<D, DEC>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) !=
        cudaSuccess)
        return MSA_ERR_CUDA;
    if (!DEC) {
        // The register split only balances if the kernel launches with
        // exactly kRegsLaunch registers per thread; otherwise a growing
        // warpgroup would wait for registers that never come.  Refuse.
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, msa_attention_kernel<D, DEC>) != cudaSuccess ||
            fa.numRegs != C::kRegsLaunch) {
            fprintf(stderr, "libmsa: attention kernel has %d registers per thread, expected %d\n", fa.numRegs,
                    C::kRegsLaunch);
            return MSA_ERR_CUDA;
        }
    }
    done.fetch_or(bit, std::memory_order_release);
    return MSA_OK;
}

template <int D, bool DEC>
static int launch_d(const msa_plan_s* P, const AttnParams& prm, const CUtensorMap* maps, cudaStream_t st) {
    using C = Cfg<D, DEC>;
    const int rc = configure_current_device<D, DEC>();
    if (rc != MSA_OK) return rc;
    // Decode-only launches use programmatic stream serialization: the launch
    // may overlap the end of the kernel before it (the kernel waits for that
    // one's results itself).  Measured on back-to-back append + attention
    // steps: 8 sequences x 128 keys 16.6 -> 12.9 us, 32 sequences at D = 64
    // 110.6 -> 106.0 us, 32 sequences of 2K-16K keys at D = 128 194.5 ->
    // 188.8 us.  Launches with prefill items run for milliseconds and keep
    // plain stream order (with the attribute and an early trigger the mixed
    // batch measured 2 % slower).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P->grid);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = DEC ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, msa_attention_kernel<D, DEC>, prm, maps[0], maps[1], maps[2],
                                             maps[3], maps[4], maps[5], maps[6], maps[7], maps[8]);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

int launch_attention(const msa_plan_s* P, const void* q, const void* k_pool, const void* v_pool,
                     int64_t pool_tokens, void* out, int32_t out_dtype, float* lse, msa_stream_t stream) {
    return launch_attention_ws(P, P->workspace, q, k_pool, v_pool, pool_tokens, out, out_dtype, lse, stream);
}

int launch_attention_ws(const msa_plan_s* P, void* workspace, const void* q, const void* k_pool,
                        const void* v_pool, int64_t pool_tokens, void* out, int32_t out_dtype, float* lse,
                        msa_stream_t stream) {
    const int D = P->dims.head_dim, Hq = P->dims.num_q_heads, Hkv = P->dims.num_kv_heads;
    CUtensorMap maps[9];
    const int64_t nq = P->info.num_q_rows;
    // K and V with boxes of 128 (a whole tile), 64, 32 and 16 rows (pieces
    // of tiles that span segments), then Q
    const int box_rows[4] = {kTileKeys, 4 * kBlock, 2 * kBlock, kBlock};
    for (int i = 0; i < 4; ++i)
        if (!make_map(&maps[i], k_pool, pool_tokens, Hkv, D, box_rows[i]) ||
            !make_map(&maps[4 + i], v_pool, pool_tokens, Hkv, D, box_rows[i]))
            return MSA_ERR_CUDA;
    if (!make_map(&maps[8], q, nq, Hq, D, kTileRows))
        return MSA_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const WsLayout& W = P->lay;
    AttnParams prm;
    prm.items = reinterpret_cast<const Item*>(ws + W.items);
    prm.groups = reinterpret_cast<const Group*>(ws + W.groups);
    prm.runs = reinterpret_cast<const Run*>(ws + W.runs);
    prm.pos = reinterpret_cast<const int32_t*>(ws + W.pos);
    prm.order = reinterpret_cast<const int32_t*>(ws + W.order);
    prm.sched = reinterpret_cast<int32_t*>(ws + W.sched);
    prm.n_items = (int32_t)P->items.size();
    prm.counters = reinterpret_cast<int32_t*>(ws + W.counters);
    prm.error_word = reinterpret_cast<int32_t*>(ws + W.error);
    prm.dec_part = reinterpret_cast<float*>(ws + W.dec_part);
    prm.dec_lse = reinterpret_cast<float*>(ws + W.dec_lse);
    prm.pre_part = reinterpret_cast<float*>(ws + W.pre_part);
    prm.pre_lse = reinterpret_cast<float*>(ws + W.pre_lse);
    prm.q = static_cast<const __nv_bfloat16*>(q);
    prm.out = out;
    prm.lse = lse;
    prm.out_fp32 = out_dtype == MSA_OUT_FP32;
    prm.Hq = Hq;
    prm.G = P->G;
    prm.has_prefill = P->info.num_prefill_items > 0;
    prm.scale_log2 = P->dims.softmax_scale * 1.4426950408889634f;
    prm.n_runs = (int32_t)P->runs.size();
    prm.limit_ns = 2000000000ull;  // 2 s per wait: far beyond any legitimate stall
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (prm.has_prefill)
        return D == 128 ? launch_d<128, false>(P, prm, maps, st) : launch_d<64, false>(P, prm, maps, st);
    return D == 128 ? launch_d<128, true>(P, prm, maps, st) : launch_d<64, true>(P, prm, maps, st);
}

}  // namespace msa
