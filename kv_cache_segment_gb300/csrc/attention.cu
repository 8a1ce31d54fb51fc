// attention.cu -- the persistent Multi-Segment Attention kernel for sm_103a.
//
// One launch serves every work item of a plan: decode groups (a sequence's
// few trailing query rows, all G query heads of one kv head packed as the
// rows of a warp-level MMA) and prefill / hole-recompute tiles (128 query
// rows of one query head, tcgen05 tensor cores with TMEM accumulators).
// Each item walks its key range segment by segment: KV tiles never cross a
// segment, so every tile is one rectangle of the paged pool fetched by TMA
// (AsymCache explainer, "核心方法 1. Multi-Segment Attention": attend to the
// physically contiguous segments of the live KV; MSA summary: one kernel over
// many disjoint segments instead of a launch per segment).  Segments of one
// item are combined by the online-softmax running (max, sum, output) state,
// which is the pairwise form of the log-sum-exp merge; items of a group that
// was split for SM balance write (output, lse) partials and the last one to
// finish merges them by log-sum-exp.
//
// CTA = 6 warps:
//   warp 0      TMA producer: Q tile (prefill) and K/V tiles into a ring of
//               shared-memory stages, one mbarrier pair per stage.
//   warp 1      owns TMEM; one lane issues tcgen05.mma: S = Q K^T into one
//               of two TMEM S buffers, then O += P V into the TMEM O buffer.
//   warps 2..5  compute: prefill softmax / epilogue (thread = tile row =
//               TMEM lane), or the decode math (mma.sync on 32 keys each).
#include <cuda.h>
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
    const int32_t* cta_indptr;
    const int32_t* cta_items;
    int32_t* counters;
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
// Q tile and no P buffer, so those bytes become extra K/V stages (more bytes
// in flight for the HBM-bound path); the decode merge scratch then has its
// own region.
template <int D, bool DEC>
struct Cfg {
    static constexpr int kPanels = D / 64;            // 64-element (128-byte) column panels
    static constexpr int kPanelBytes = 128 * 128;     // one panel of a 128-row tile
    static constexpr int kTileBytes = kPanels * kPanelBytes;  // 128 rows x D bf16
    static constexpr int kStages = DEC ? (D == 128 ? 3 : 6) : (D == 128 ? 2 : 4);
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = DEC ? 0 : kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffP = kOffV + kStages * kTileBytes;  // P buffer, or the decode scratch
    static constexpr int kScratchBytes = 4 * kDecRows * D * 4;
    static constexpr int kPBytes = DEC ? kScratchBytes : 2 * kPanelBytes;  // P: 128 rows x 128 keys bf16
    static constexpr int kOffCtl = kOffP + kPBytes;
    static constexpr int kCtlBytes = 1536;
    static constexpr int kSmem = kOffCtl + kCtlBytes + 1024;  // + slack to align the base to 1024
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmemO = 256;           // S buffers at columns 0 and 128
    static_assert(kScratchBytes <= kPBytes, "decode merge scratch must fit");
    static_assert(kSmem + 64 <= 232448, "shared memory over the per-CTA limit");
};

struct Ctl {
    uint64_t k_full[8], k_empty[8], v_full[8], v_empty[8];
    uint64_t q_full, q_empty;
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full, p_empty, o_full, o_empty;
    uint64_t drain;
    uint64_t csync;  // bounded barrier of the 128 compute threads
    int4 meta[8];  // per stage: first logical key, valid keys, item, unused
    uint32_t tmem_base;
    int abort;
    int flag_last;
    int pad;
    float dec_m[4][kDecRows];
    float dec_l[4][kDecRows];
    float dec_lr[4][kDecRows];
};

static_assert(sizeof(Ctl) <= Cfg<128, false>::kCtlBytes, "control block too large");

constexpr int kThreads = 192;
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

// Sum of the two bf16 values packed in w, as fp32 (exact).
__device__ __forceinline__ float bf16x2_sum(uint32_t w) {
    return __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
}

// Barrier of the 128 compute threads built on an mbarrier, so that a wait
// that can never complete (a warp gave up on a timeout) runs out instead of
// hanging.  `cnt` counts this thread's passes.
__device__ __forceinline__ bool compute_sync(const AttnParams& p, Ctl* ctl, uint32_t& cnt) {
    ptx::mbar_arrive(&ctl->csync);
    const bool ok = wait_bar(p, ctl, &ctl->csync, cnt & 1, kErrTimeoutCompute);
    ++cnt;
    return ok;
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

template <int D, bool DEC>
__device__ void producer(const AttnParams& p, uint8_t* smem, Ctl* ctl, int i0, int i1, const CUtensorMap* tmK,
                         const CUtensorMap* tmK16, const CUtensorMap* tmV, const CUtensorMap* tmV16,
                         const CUtensorMap* tmQ) {
    using C = Cfg<D, DEC>;
    uint32_t kv_cnt = 0, q_cnt = 0;
    for (int ii = i0; ii < i1; ++ii) {
        const Item it = p.items[p.cta_items[ii]];
        const Group g = p.groups[it.group];
        int kvh = g.head;
        if (it.kind == kPrefill) {
            kvh = g.head / p.G;
            if (!wait_bar(p, ctl, &ctl->q_empty, (q_cnt & 1) ^ 1, kErrTimeoutProducer)) goto drain;
            ptx::mbar_arrive_expect_tx(&ctl->q_full, C::kTileBytes);
            for (int pn = 0; pn < C::kPanels; ++pn)
                ptx::tma_load_3d(smem + C::kOffQ + pn * C::kPanelBytes, tmQ, pn * 64, g.head, g.row0, &ctl->q_full);
            ++q_cnt;
        }
        // KV tiles are 128-key windows of the item's logical key range.  A
        // window that lies inside one segment is one TMA rectangle; where it
        // spans segments, each piece is fetched from its own segment, one
        // 16-row box per block (segments are whole blocks, so every piece is).
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
            if (!wait_bar(p, ctl, &ctl->k_empty[st], ph ^ 1, kErrTimeoutProducer)) goto drain;
            if (!wait_bar(p, ctl, &ctl->v_empty[st], ph ^ 1, kErrTimeoutProducer)) goto drain;
            ctl->meta[st] = make_int4(t0, n, ii, 0);
            uint8_t* ks = smem + C::kOffK + st * C::kTileBytes;
            uint8_t* vs = smem + C::kOffV + st * C::kTileBytes;
            const uint32_t bytes = (uint32_t)(((n + kBlock - 1) & ~(kBlock - 1)) * D * 2);
            ptx::mbar_arrive_expect_tx(&ctl->k_full[st], bytes);
            ptx::mbar_arrive_expect_tx(&ctl->v_full[st], bytes);
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
                    for (int pn = 0; pn < C::kPanels; ++pn) {
                        ptx::tma_load_3d(ks + pn * C::kPanelBytes, tmK, pn * 64, kvh, phys, &ctl->k_full[st]);
                        ptx::tma_load_3d(vs + pn * C::kPanelBytes, tmV, pn * 64, kvh, phys, &ctl->v_full[st]);
                    }
                } else {
                    const int nb = (pend - cur + kBlock - 1) / kBlock;
                    for (int b = 0; b < nb; ++b)
                        for (int pn = 0; pn < C::kPanels; ++pn) {
                            const int so = pn * C::kPanelBytes + (off + b * kBlock) * 128;
                            ptx::tma_load_3d(ks + so, tmK16, pn * 64, kvh, phys + b * kBlock, &ctl->k_full[st]);
                            ptx::tma_load_3d(vs + so, tmV16, pn * 64, kvh, phys + b * kBlock, &ctl->v_full[st]);
                        }
                }
                cur = pend;
            }
            ++kv_cnt;
        }
    }
drain:
    // Wait (bounded, ignoring the abort flag) for the loads still in flight,
    // so that none lands in shared memory after the CTA has exited.
    {
        static __shared__ int never;  // an abort flag nobody sets
        never = 0;
        const uint32_t tail = kv_cnt < (uint32_t)C::kStages ? kv_cnt : (uint32_t)C::kStages;
        for (uint32_t k = kv_cnt - tail; k < kv_cnt; ++k) {
            const int st = k % C::kStages;
            const uint32_t ph = (k / C::kStages) & 1;
            ptx::mbar_wait(&ctl->k_full[st], ph, &never, 100000000ull);
            ptx::mbar_wait(&ctl->v_full[st], ph, &never, 100000000ull);
        }
        if (q_cnt > 0) ptx::mbar_wait(&ctl->q_full, (q_cnt - 1) & 1, &never, 100000000ull);
    }
}

// ------------------------------------------------------------ MMA warp --

template <int D, bool DEC>
__device__ void mma_issuer(const AttnParams& p, uint8_t* smem, Ctl* ctl, int i0, int i1) {
    using C = Cfg<D, DEC>;
    constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, 128, 0, 0);  // Q K-major, K K-major
    constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, D, 0, 1);   // P K-major, V MN-major
    const uint32_t tbase = ctl->tmem_base;
    const uint32_t sQ = ptx::smem_u32(smem + C::kOffQ);
    const uint32_t sK = ptx::smem_u32(smem + C::kOffK);
    const uint32_t sV = ptx::smem_u32(smem + C::kOffV);
    const uint32_t sP = ptx::smem_u32(smem + C::kOffP);
    uint32_t kv_cnt = 0, q_cnt = 0, s_cnt = 0, pv_cnt = 0, o_cnt = 0;
    for (int ii = i0; ii < i1; ++ii) {
        const Item it = p.items[p.cta_items[ii]];
        const int T = it.pad;  // KV tiles of this item
        if (it.kind != kPrefill) { kv_cnt += T; continue; }
        const int pmin = p.pos[p.groups[it.group].row0];  // rows ascend: the tile's smallest position
        if (!wait_bar(p, ctl, &ctl->q_full, q_cnt & 1, kErrTimeoutMma)) goto drain;
        ++q_cnt;
        for (int j = 0; j <= T; ++j) {
            if (j < T) {
                const uint32_t k = kv_cnt + j;
                const int st = k % C::kStages;
                const uint32_t ph = (k / C::kStages) & 1;
                if (!wait_bar(p, ctl, &ctl->k_full[st], ph, kErrTimeoutMma)) goto drain;
                const int sb = s_cnt & 1;
                if (!wait_bar(p, ctl, &ctl->s_empty[sb], ((s_cnt >> 1) & 1) ^ 1, kErrTimeoutMma)) goto drain;
                ptx::tc_fence_after();
                const uint32_t kbase = sK + st * C::kTileBytes;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::kPanelBytes + (ks & 3) * 32;
                    const uint64_t ad = ptx::smem_desc(sQ + off, 16, 1024, 2);
                    const uint64_t bd = ptx::smem_desc(kbase + off, 16, 1024, 2);
                    ptx::tc_mma_ss(tbase + sb * 128, ad, bd, kIdescS, ks > 0);
                }
                ptx::tc_commit(&ctl->k_empty[st]);
                ptx::tc_commit(&ctl->s_full[sb]);
                ++s_cnt;
                if (j == T - 1) ptx::tc_commit(&ctl->q_empty);
            }
            if (j >= 1) {
                const int jj = j - 1;
                const uint32_t k = kv_cnt + jj;
                const int st = k % C::kStages;
                const uint32_t ph = (k / C::kStages) & 1;
                if (!wait_bar(p, ctl, &ctl->p_full, pv_cnt & 1, kErrTimeoutMma)) goto drain;
                if (!wait_bar(p, ctl, &ctl->v_full[st], ph, kErrTimeoutMma)) goto drain;
                if (jj == 0 && !wait_bar(p, ctl, &ctl->o_empty, (o_cnt & 1) ^ 1, kErrTimeoutMma)) goto drain;
                ptx::tc_fence_after();
                const int4 mt = ctl->meta[st];
                const int nk = (mt.y + 15) >> 4;
                const uint32_t vbase = sV + st * C::kTileBytes;
                // rows that see fewer than 128 keys get a second pass with the
                // bf16 residual of P (see prefill_item)
                const bool precise = mt.x < kTileKeys && pmin < kTileKeys;
                for (int pass = 0; pass < (precise ? 2 : 1); ++pass) {
                    if (pass == 1) {
                        if (!wait_bar(p, ctl, &ctl->p_full, pv_cnt & 1, kErrTimeoutMma)) goto drain;
                        ptx::tc_fence_after();
                    }
                    for (int ks = 0; ks < nk; ++ks) {
                        const uint64_t ad =
                            ptx::smem_desc(sP + (ks >> 2) * C::kPanelBytes + (ks & 3) * 32, 16, 1024, 2);
                        const uint64_t bd = ptx::smem_desc(vbase + ks * 16 * 128, C::kPanelBytes, 1024, 2);
                        ptx::tc_mma_ss(tbase + C::kTmemO, ad, bd, kIdescPV, (jj > 0 || ks > 0 || pass > 0) ? 1u : 0u);
                    }
                    ptx::tc_commit(&ctl->p_empty);
                    ++pv_cnt;
                }
                ptx::tc_commit(&ctl->v_empty[st]);
                if (jj == T - 1) {
                    ptx::tc_commit(&ctl->o_full);
                    ++o_cnt;
                }
            }
        }
        kv_cnt += T;
    }
drain:
    return;
}

// ----------------------------------------------------- output helpers --

__device__ __forceinline__ void store_out(const AttnParams& p, int64_t idx, float v) {
    if (p.out_fp32) static_cast<float*>(p.out)[idx] = v;
    else static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
}

// ------------------------------------------------------ decode (compute) --

template <int D, bool DEC>
__device__ bool decode_item(const AttnParams& p, uint8_t* smem, Ctl* ctl, const Item& it, const Group& g,
                            uint32_t& kv_cnt, uint32_t& cs, int cw, int lane) {
    using C = Cfg<D, DEC>;
    constexpr int KS = D / 16;  // k-steps over the head dimension
    constexpr int NT = D / 8;   // 8-column output tiles
    const int G = p.G;
    const int M = g.nrows * G;
    const int kvh = g.head;
    const int gr = lane >> 2, tq = lane & 3;

    const int prow0 = gr < M ? p.pos[g.row0 + gr / G] : -1;
    const int prow1 = gr + 8 < M ? p.pos[g.row0 + (gr + 8) / G] : -1;

    // Q fragments (rows = query row x head, zero past M)
    uint32_t qa[KS][4];
    {
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(p.q);
        auto qword = [&](int m, int dim) -> uint32_t {
            if (m >= M) return 0u;
            const int64_t row = g.row0 + m / G;
            const int64_t h = (int64_t)kvh * G + m % G;
            return qw[((row * p.Hq + h) * D + dim) >> 1];
        };
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qa[ks][0] = qword(gr, ks * 16 + 2 * tq);
            qa[ks][1] = qword(gr + 8, ks * 16 + 2 * tq);
            qa[ks][2] = qword(gr, ks * 16 + 8 + 2 * tq);
            qa[ks][3] = qword(gr + 8, ks * 16 + 8 + 2 * tq);
        }
    }

    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    // lrun: fp32 probability sums (lse); rrun: sums of the bf16-rounded
    // probabilities the PV MMA consumes (output normaliser)
    float mrun0 = -INFINITY, mrun1 = -INFINITY, lrun0 = 0.f, lrun1 = 0.f, rrun0 = 0.f, rrun1 = 0.f;
    const int key0 = cw * 32;
    const int T = it.pad;

    for (int t = 0; t < T; ++t) {
        const uint32_t k = kv_cnt + t;
        const int st = k % C::kStages;
        const uint32_t ph = (k / C::kStages) & 1;
        if (!wait_bar(p, ctl, &ctl->k_full[st], ph, kErrTimeoutCompute)) return false;
        if (!wait_bar(p, ctl, &ctl->v_full[st], ph, kErrTimeoutCompute)) return false;
        const int4 mt = ctl->meta[st];
        const int kt0 = mt.x, n = mt.y;
        if (key0 < n) {
            const uint32_t kb = ptx::smem_u32(smem + C::kOffK + st * C::kTileBytes);
            const uint32_t vb = ptx::smem_u32(smem + C::kOffV + st * C::kTileBytes);
            float s[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
                const int key = key0 + nt * 8 + (lane & 7);
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk) {
                    uint32_t b0, b1, b2, b3;
                    ptx::ldmatrix_x4(kb + sw128_off<D>(key, kk * 4 + (lane >> 3)), b0, b1, b2, b3);
                    ptx::mma_bf16_16816(s[nt], qa[2 * kk], b0, b1);
                    ptx::mma_bf16_16816(s[nt], qa[2 * kk + 1], b2, b3);
                }
            }
            // mask (key inside the tile, causal key <= row position), scale to log2 units
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
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
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(mrun0, mx0), mn1 = fmaxf(mrun1, mx1);
            const float use0 = mn0 == -INFINITY ? 0.f : mn0;
            const float use1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = ptx::ex2(mrun0 - use0), al1 = ptx::ex2(mrun1 - use1);
            mrun0 = mn0;
            mrun1 = mn1;
            float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                s[nt][0] = ptx::ex2(s[nt][0] - use0);
                s[nt][1] = ptx::ex2(s[nt][1] - use0);
                s[nt][2] = ptx::ex2(s[nt][2] - use1);
                s[nt][3] = ptx::ex2(s[nt][3] - use1);
                sum0 += s[nt][0] + s[nt][1];
                sum1 += s[nt][2] + s[nt][3];
            }
            lrun0 = lrun0 * al0 + sum0;
            lrun1 = lrun1 * al1 + sum1;
            rrun0 *= al0;
            rrun1 *= al1;
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    o[i][0] *= al0; o[i][1] *= al0;
                    o[i][2] *= al1; o[i][3] *= al1;
                }
            }
            const bool tail = key0 + 32 > n;
#pragma unroll
            for (int kst = 0; kst < 2; ++kst) {
                uint32_t a[4];
                a[0] = ptx::pack_bf16x2(s[2 * kst][0], s[2 * kst][1]);
                a[1] = ptx::pack_bf16x2(s[2 * kst][2], s[2 * kst][3]);
                a[2] = ptx::pack_bf16x2(s[2 * kst + 1][0], s[2 * kst + 1][1]);
                a[3] = ptx::pack_bf16x2(s[2 * kst + 1][2], s[2 * kst + 1][3]);
                const int kbase = key0 + kst * 16;
                if (kbase >= n) break;
                rrun0 += bf16x2_sum(a[0]) + bf16x2_sum(a[2]);
                rrun1 += bf16x2_sum(a[1]) + bf16x2_sum(a[3]);
                // keys below 128: rows may see few keys, add the bf16 residual
                // of P as a second MMA (see prefill_item)
                const bool precise = kt0 < kTileKeys;
                uint32_t alo[4] = {0u, 0u, 0u, 0u};
                if (precise) {
                    alo[0] = ptx::pack_bf16x2(s[2 * kst][0] - __uint_as_float(a[0] << 16),
                                              s[2 * kst][1] - __uint_as_float(a[0] & 0xffff0000u));
                    alo[1] = ptx::pack_bf16x2(s[2 * kst][2] - __uint_as_float(a[1] << 16),
                                              s[2 * kst][3] - __uint_as_float(a[1] & 0xffff0000u));
                    alo[2] = ptx::pack_bf16x2(s[2 * kst + 1][0] - __uint_as_float(a[2] << 16),
                                              s[2 * kst + 1][1] - __uint_as_float(a[2] & 0xffff0000u));
                    alo[3] = ptx::pack_bf16x2(s[2 * kst + 1][2] - __uint_as_float(a[3] << 16),
                                              s[2 * kst + 1][3] - __uint_as_float(a[3] & 0xffff0000u));
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
                    if (precise) {
                        ptx::mma_bf16_16816(o[2 * dp], alo, b0 & m0, b1 & m1);
                        ptx::mma_bf16_16816(o[2 * dp + 1], alo, b2 & m0, b3 & m1);
                    }
                }
            }
        }
        if (!compute_sync(p, ctl, cs)) return false;
        if (cw == 0 && lane == 0) {
            ptx::mbar_arrive(&ctl->k_empty[st]);
            ptx::mbar_arrive(&ctl->v_empty[st]);
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
    float* scr = reinterpret_cast<float*>(smem + C::kOffP);  // [4][16][D]
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
    if (!compute_sync(p, ctl, cs)) return false;
    const int tid = cw * 32 + lane;
    const bool split = g.n_parts > 1;
    float* part = split ? p.dec_part + (int64_t)(g.slot + it.part) * kDecRows * D : nullptr;
    float* plse = split ? p.dec_lse + (int64_t)(g.slot + it.part) * kDecRows : nullptr;
    for (int e = tid; e < M * D; e += 128) {
        const int m = e / D, d = e % D;
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) mm = fmaxf(mm, ctl->dec_m[w][m]);
        float val = 0.f, lse2 = -INFINITY;
        if (mm != -INFINITY) {
            float L = 0.f, LR = 0.f, acc = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float f = ptx::ex2(ctl->dec_m[w][m] - mm);
                L += ctl->dec_l[w][m] * f;
                LR += ctl->dec_lr[w][m] * f;
                acc += scr[(w * kDecRows + m) * D + d] * f;
            }
            val = acc / LR;
            lse2 = mm + log2f(L);
        }
        if (split) {
            part[m * D + d] = val;
            if (d == 0) plse[m] = lse2;
        } else {
            const int64_t row = g.row0 + m / G;
            const int64_t h = (int64_t)kvh * G + m % G;
            store_out(p, (row * p.Hq + h) * D + d, val);
            if (d == 0 && p.lse) p.lse[row * p.Hq + h] = lse2 * kLn2;
        }
    }
    if (split) {
        __threadfence();
        if (!compute_sync(p, ctl, cs)) return false;
        if (tid == 0) {
            const int old = atomicAdd(&p.counters[it.group], 1);
            ctl->flag_last = (old == g.n_parts - 1);
        }
        if (!compute_sync(p, ctl, cs)) return false;
        if (ctl->flag_last) {
            __threadfence();
            const float* base = p.dec_part + (int64_t)g.slot * kDecRows * D;
            const float* lbase = p.dec_lse + (int64_t)g.slot * kDecRows;
            for (int e = tid; e < M * D; e += 128) {
                const int m = e / D, d = e % D;
                float mm = -INFINITY;
                for (int q = 0; q < g.n_parts; ++q) mm = fmaxf(mm, __ldcg(lbase + q * kDecRows + m));
                float val = 0.f, lse2 = -INFINITY;
                if (mm != -INFINITY) {
                    float L = 0.f, acc = 0.f;
                    for (int q = 0; q < g.n_parts; ++q) {
                        const float f = ptx::ex2(__ldcg(lbase + q * kDecRows + m) - mm);
                        L += f;
                        acc += f * __ldcg(base + ((int64_t)q * kDecRows + m) * D + d);
                    }
                    val = acc / L;
                    lse2 = mm + log2f(L);
                }
                const int64_t row = g.row0 + m / G;
                const int64_t h = (int64_t)kvh * G + m % G;
                store_out(p, (row * p.Hq + h) * D + d, val);
                if (d == 0 && p.lse) p.lse[row * p.Hq + h] = lse2 * kLn2;
            }
            if (tid == 0) p.counters[it.group] = 0;  // ready for the next launch
        }
    }
    return compute_sync(p, ctl, cs);  // scratch and flag free for the next item
}

// ----------------------------------------------------- prefill (compute) --

template <int D, bool DEC>
__device__ bool prefill_item(const AttnParams& p, uint8_t* smem, Ctl* ctl, const Item& it, const Group& g,
                             uint32_t& kv_cnt, uint32_t& s_cnt, uint32_t& pvb, uint32_t& o_cnt, uint32_t& cs,
                             int cw, int warp, int lane) {
    using C = Cfg<D, DEC>;
    const int quarter = warp & 3;
    const int ri = quarter * 32 + lane;  // tile row = TMEM lane
    const bool valid = ri < g.nrows;
    const int prow = valid ? p.pos[g.row0 + ri] : -1;
    const int pmin = p.pos[g.row0];
    const uint32_t tlane = ctl->tmem_base + ((uint32_t)(quarter * 32) << 16);
    uint8_t* pbuf = smem + C::kOffP;
    const int T = it.pad;
    // l: sum of the fp32 probabilities (gives lse); lr: sum of the same
    // values rounded to bf16, exactly as the PV MMA consumes them (the
    // normaliser of the output, so that out is a true weighted mean of V
    // rows even when one key dominates)
    float m = -INFINITY, l = 0.f, lr = 0.f;

    for (int j = 0; j < T; ++j) {
        const uint32_t k = kv_cnt + j;
        const int st = k % C::kStages;
        const uint32_t ph = (k / C::kStages) & 1;
        const int sb = s_cnt & 1;
        if (!wait_bar(p, ctl, &ctl->s_full[sb], (s_cnt >> 1) & 1, kErrTimeoutCompute)) return false;
        if (!wait_bar(p, ctl, &ctl->k_full[st], ph, kErrTimeoutCompute)) return false;
        ptx::tc_fence_after();
        const int4 mt = ctl->meta[st];
        const int kt0 = mt.x, n = mt.y;
        // rows that see fewer than 128 keys in total get a second PV pass
        // with the bf16 residual of P (see below); those tiles keep their S
        // buffer until the second pass has re-read it
        const bool precise = kt0 < kTileKeys && pmin < kTileKeys;
        float s[128];
        ptx::tmem_ld128(tlane + sb * 128, s);
        if (!precise) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(&ctl->s_empty[sb]);
        }
        ++s_cnt;

        const int lim = max(0, min(n, prow - kt0 + 1));  // visible columns of this row
        float mx;
        {
            // eight independent chains, then a tree: no 128-long dependency
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; ++c) m8[c & 7] = fmaxf(m8[c & 7], c < lim ? s[c] : -INFINITY);
            mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        }
        float alpha = 1.f;
        bool resc = false;
        if (lim > 0) {
            const float ms = mx * p.scale_log2;
            // keep the running max unless the new one is larger by more than
            // 8 (log2 units): values stay <= 256, rescales become rare
            if (ms > m + 8.f) {
                alpha = ptx::ex2(m - ms);
                resc = j > 0;
                m = ms;
            }
        }
        // previous PV batches done: the P buffer is free and O is current
        if (j > 0 && !wait_bar(p, ctl, &ctl->p_empty, (pvb - 1) & 1, kErrTimeoutCompute)) return false;
        if (__any_sync(0xffffffffu, resc)) {
            ptx::tc_fence_after();
            const float f = resc ? alpha : 1.f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                float ov[32];
                ptx::tmem_ld32(tlane + C::kTmemO + c * 32, ov);
#pragma unroll
                for (int i = 0; i < 32; ++i) ov[i] *= f;
                ptx::tmem_st32(tlane + C::kTmemO + c * 32, ov);
            }
            ptx::tmem_wait_st();
        }
        float sum4[4] = {0.f, 0.f, 0.f, 0.f}, sr4[4] = {0.f, 0.f, 0.f, 0.f};
        const float sl = p.scale_log2;
#pragma unroll
        for (int c8 = 0; c8 < 16; ++c8) {
            float pv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int c = c8 * 8 + e;
                pv[e] = c < lim ? ptx::ex2(fmaf(s[c], sl, -m)) : 0.f;
                sum4[e & 3] += pv[e];
            }
            uint4 w;
            w.x = ptx::pack_bf16x2(pv[0], pv[1]);
            w.y = ptx::pack_bf16x2(pv[2], pv[3]);
            w.z = ptx::pack_bf16x2(pv[4], pv[5]);
            w.w = ptx::pack_bf16x2(pv[6], pv[7]);
            sr4[c8 & 3] += (bf16x2_sum(w.x) + bf16x2_sum(w.y)) + (bf16x2_sum(w.z) + bf16x2_sum(w.w));
            const int panel = c8 >> 3, cc = c8 & 7;
            *reinterpret_cast<uint4*>(pbuf + panel * C::kPanelBytes + ri * 128 + ((cc ^ (ri & 7)) << 4)) = w;
        }
        const float sum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
        float sumr = (sr4[0] + sr4[1]) + (sr4[2] + sr4[3]);
        l = l * alpha + sum;
        lr = lr * alpha;
        if (n & (kBlock - 1)) {
            // The tile ends inside the sequence's last, partial block: rows
            // [n, ceil16(n)) of the V stage are pool rows past L_s and may
            // hold anything.  The PV MMA covers whole 16-row steps, so zero
            // them (P is already 0 there).
            if (!wait_bar(p, ctl, &ctl->v_full[st], ph, kErrTimeoutCompute)) return false;
            const int nz = ((n + 15) & ~15) - n;
            uint8_t* vs = smem + C::kOffV + st * C::kTileBytes;
            const int chunks = nz * (D / 8);
            for (int c = cw * 32 + lane; c < chunks; c += 128) {
                const int r = n + c / (D / 8), cc = c % (D / 8);
                *reinterpret_cast<uint4*>(vs + (cc >> 3) * C::kPanelBytes + r * 128 + (cc & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(&ctl->p_full);
        ++pvb;
        if (precise) {
            // Rows of this tile see fewer than 128 keys in total, so a bf16
            // rounding of one probability is not averaged away (the output
            // error would be ~2^-9 * |V|).  Second pass: the bf16 residual
            // p - bf16(p), accumulated by a second PV MMA once the first
            // one has released the P buffer.  p is recomputed from S.
            if (!wait_bar(p, ctl, &ctl->p_empty, (pvb - 1) & 1, kErrTimeoutCompute)) return false;
            float s2[128];
            ptx::tmem_ld128(tlane + sb * 128, s2);
            ptx::tc_fence_before();
            ptx::mbar_arrive(&ctl->s_empty[sb]);
            float sumlo = 0.f;
#pragma unroll
            for (int c8 = 0; c8 < 16; ++c8) {
                uint32_t wv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = c8 * 8 + 2 * e;
                    const float a = c < lim ? ptx::ex2(fmaf(s2[c], sl, -m)) : 0.f;
                    const float b = c + 1 < lim ? ptx::ex2(fmaf(s2[c + 1], sl, -m)) : 0.f;
                    const uint32_t hi = ptx::pack_bf16x2(a, b);
                    wv[e] = ptx::pack_bf16x2(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xffff0000u));
                    sumlo += bf16x2_sum(wv[e]);
                }
                const int panel = c8 >> 3, cc = c8 & 7;
                *reinterpret_cast<uint4*>(pbuf + panel * C::kPanelBytes + ri * 128 + ((cc ^ (ri & 7)) << 4)) =
                    make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
            sumr += sumlo;
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&ctl->p_full);
            ++pvb;
        }
        lr += sumr;
    }
    kv_cnt += T;

    // epilogue
    if (!wait_bar(p, ctl, &ctl->o_full, o_cnt & 1, kErrTimeoutCompute)) return false;
    ++o_cnt;
    ptx::tc_fence_after();
    float ov[D];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) ptx::tmem_ld32(tlane + C::kTmemO + c * 32, ov + c * 32);
    ptx::tc_fence_before();
    ptx::mbar_arrive(&ctl->o_empty);

    const float inv = lr > 0.f ? 1.f / lr : 0.f;
    const float lse2 = l > 0.f ? m + log2f(l) : -INFINITY;
    const int tid = cw * 32 + lane;
    if (g.n_parts == 1) {
        if (valid) {
            const int64_t base = ((int64_t)(g.row0 + ri) * p.Hq + g.head) * D;
            if (p.out_fp32) {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + base);
#pragma unroll
                for (int c = 0; c < D / 4; ++c)
                    dst[c] = make_float4(ov[4 * c] * inv, ov[4 * c + 1] * inv, ov[4 * c + 2] * inv, ov[4 * c + 3] * inv);
            } else {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + base);
#pragma unroll
                for (int c = 0; c < D / 8; ++c) {
                    uint4 w;
                    w.x = ptx::pack_bf16x2(ov[8 * c] * inv, ov[8 * c + 1] * inv);
                    w.y = ptx::pack_bf16x2(ov[8 * c + 2] * inv, ov[8 * c + 3] * inv);
                    w.z = ptx::pack_bf16x2(ov[8 * c + 4] * inv, ov[8 * c + 5] * inv);
                    w.w = ptx::pack_bf16x2(ov[8 * c + 6] * inv, ov[8 * c + 7] * inv);
                    dst[c] = w;
                }
            }
            if (p.lse) p.lse[(int64_t)(g.row0 + ri) * p.Hq + g.head] = lse2 * kLn2;
        }
        return true;
    }
    // split group: write this part, the last part to arrive merges
    {
        float* part = p.pre_part + ((int64_t)(g.slot + it.part) * kTileRows + ri) * D;
        float4* dst = reinterpret_cast<float4*>(part);
#pragma unroll
        for (int c = 0; c < D / 4; ++c)
            dst[c] = make_float4(ov[4 * c] * inv, ov[4 * c + 1] * inv, ov[4 * c + 2] * inv, ov[4 * c + 3] * inv);
        p.pre_lse[(int64_t)(g.slot + it.part) * kTileRows + ri] = lse2;
    }
    __threadfence();
    if (!compute_sync(p, ctl, cs)) return false;
    if (tid == 0) {
        const int old = atomicAdd(&p.counters[it.group], 1);
        ctl->flag_last = (old == g.n_parts - 1);
    }
    if (!compute_sync(p, ctl, cs)) return false;
    if (ctl->flag_last) {
        __threadfence();
        if (valid) {
            float mm = -INFINITY;
            for (int q = 0; q < g.n_parts; ++q)
                mm = fmaxf(mm, __ldcg(p.pre_lse + (int64_t)(g.slot + q) * kTileRows + ri));
            float L = 0.f;
            float acc[D];
#pragma unroll
            for (int d = 0; d < D; ++d) acc[d] = 0.f;
            if (mm != -INFINITY) {
                for (int q = 0; q < g.n_parts; ++q) {
                    const float f = ptx::ex2(__ldcg(p.pre_lse + (int64_t)(g.slot + q) * kTileRows + ri) - mm);
                    L += f;
                    const float4* src =
                        reinterpret_cast<const float4*>(p.pre_part + ((int64_t)(g.slot + q) * kTileRows + ri) * D);
#pragma unroll
                    for (int c = 0; c < D / 4; ++c) {
                        const float4 v = __ldcg(src + c);
                        acc[4 * c] += f * v.x; acc[4 * c + 1] += f * v.y;
                        acc[4 * c + 2] += f * v.z; acc[4 * c + 3] += f * v.w;
                    }
                }
            }
            const float invL = L > 0.f ? 1.f / L : 0.f;
            const int64_t base = ((int64_t)(g.row0 + ri) * p.Hq + g.head) * D;
#pragma unroll
            for (int d = 0; d < D; ++d) store_out(p, base + d, acc[d] * invL);
            if (p.lse) p.lse[(int64_t)(g.row0 + ri) * p.Hq + g.head] = L > 0.f ? (mm + log2f(L)) * kLn2 : -INFINITY;
        }
        if (tid == 0) p.counters[it.group] = 0;
    }
    return compute_sync(p, ctl, cs);
}

template <int D, bool DEC>
__device__ void compute(const AttnParams& p, uint8_t* smem, Ctl* ctl, int i0, int i1, int warp, int lane) {
    const int cw = warp - 2;
    uint32_t kv_cnt = 0, s_cnt = 0, pvb = 0, o_cnt = 0, cs = 0;
    for (int ii = i0; ii < i1; ++ii) {
        const Item it = p.items[p.cta_items[ii]];
        const Group g = p.groups[it.group];
        bool ok;
        if constexpr (DEC) {
            ok = decode_item<D, DEC>(p, smem, ctl, it, g, kv_cnt, cs, cw, lane);
        } else {
            ok = it.kind == kDecode ? decode_item<D, DEC>(p, smem, ctl, it, g, kv_cnt, cs, cw, lane)
                                    : prefill_item<D, DEC>(p, smem, ctl, it, g, kv_cnt, s_cnt, pvb, o_cnt, cs, cw,
                                                           warp, lane);
        }
        if (!ok) return;
    }
}

template <int D, bool DEC>
__global__ void __launch_bounds__(kThreads, 1)
    msa_attention_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmK16, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmV16, const __grid_constant__ CUtensorMap tmQ) {
    using C = Cfg<D, DEC>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + C::kOffCtl);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 8; ++s) {
            ptx::mbar_init(&ctl->k_full[s], 1);
            ptx::mbar_init(&ctl->k_empty[s], 1);
            ptx::mbar_init(&ctl->v_full[s], 1);
            ptx::mbar_init(&ctl->v_empty[s], 1);
        }
        ptx::mbar_init(&ctl->q_full, 1);
        ptx::mbar_init(&ctl->q_empty, 1);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&ctl->s_full[s], 1);
            ptx::mbar_init(&ctl->s_empty[s], 128);
        }
        ptx::mbar_init(&ctl->p_full, 128);
        ptx::mbar_init(&ctl->p_empty, 1);
        ptx::mbar_init(&ctl->o_full, 1);
        ptx::mbar_init(&ctl->o_empty, 128);
        ptx::mbar_init(&ctl->drain, 1);
        ptx::mbar_init(&ctl->csync, 128);
        ctl->abort = 0;
        ctl->flag_last = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmK16);
        ptx::prefetch_tmap(&tmV);
        ptx::prefetch_tmap(&tmV16);
        ptx::prefetch_tmap(&tmQ);
    }
    if (!DEC && warp == 1 && p.has_prefill) {
        ptx::tmem_alloc(&ctl->tmem_base, C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    const int i0 = p.cta_indptr[blockIdx.x], i1 = p.cta_indptr[blockIdx.x + 1];
    if (warp == 0) {
        if (lane == 0) producer<D, DEC>(p, smem, ctl, i0, i1, &tmK, &tmK16, &tmV, &tmV16, &tmQ);
    } else if (warp == 1) {
        if constexpr (!DEC) {
            if (lane == 0 && p.has_prefill) {
            mma_issuer<D, DEC>(p, smem, ctl, i0, i1);
            // every MMA issued must have completed before TMEM is released
            ptx::tc_commit(&ctl->drain);
            ptx::mbar_wait(&ctl->drain, 0, &ctl->abort, p.limit_ns);
            }
        }
    } else {
        compute<D, DEC>(p, smem, ctl, i0, i1, warp, lane);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (!DEC && warp == 1 && p.has_prefill) ptx::tmem_dealloc(ctl->tmem_base, C::kTmemCols);
}

// ------------------------------------------------------------ host side --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 3-D bf16 map over [rows, heads, D] (innermost D), box = 64 x 1 x box_rows,
// 128-byte swizzle; rows past the end read as zero.
static bool make_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int D, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool DEC>
static int launch_d(const msa_plan_s* P, const AttnParams& prm, const CUtensorMap* maps, cudaStream_t st) {
    using C = Cfg<D, DEC>;
    static bool configured = false;
    if (!configured) {
        if (cudaFuncSetAttribute(msa_attention_kernel<D, DEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmem) != cudaSuccess)
            return MSA_ERR_CUDA;
        configured = true;
    }
    msa_attention_kernel<D, DEC>
        <<<P->grid, kThreads, C::kSmem, st>>>(prm, maps[0], maps[1], maps[2], maps[3], maps[4]);
    return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

int launch_attention(const msa_plan_s* P, const void* q, const void* k_pool, const void* v_pool,
                     int64_t pool_tokens, void* out, int32_t out_dtype, float* lse, msa_stream_t stream) {
    return launch_attention_ws(P, P->workspace, q, k_pool, v_pool, pool_tokens, out, out_dtype, lse, stream);
}

int launch_attention_ws(const msa_plan_s* P, void* workspace, const void* q, const void* k_pool,
                        const void* v_pool, int64_t pool_tokens, void* out, int32_t out_dtype, float* lse,
                        msa_stream_t stream) {
    const int D = P->dims.head_dim, Hq = P->dims.num_q_heads, Hkv = P->dims.num_kv_heads;
    CUtensorMap maps[5];
    const int64_t nq = P->info.num_q_rows;
    if (!make_map(&maps[0], k_pool, pool_tokens, Hkv, D, kTileKeys) ||
        !make_map(&maps[1], k_pool, pool_tokens, Hkv, D, kBlock) ||
        !make_map(&maps[2], v_pool, pool_tokens, Hkv, D, kTileKeys) ||
        !make_map(&maps[3], v_pool, pool_tokens, Hkv, D, kBlock) ||
        !make_map(&maps[4], q, nq, Hq, D, kTileRows))
        return MSA_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const WsLayout& W = P->lay;
    AttnParams prm;
    prm.items = reinterpret_cast<const Item*>(ws + W.items);
    prm.groups = reinterpret_cast<const Group*>(ws + W.groups);
    prm.runs = reinterpret_cast<const Run*>(ws + W.runs);
    prm.pos = reinterpret_cast<const int32_t*>(ws + W.pos);
    prm.cta_indptr = reinterpret_cast<const int32_t*>(ws + W.cta_indptr);
    prm.cta_items = reinterpret_cast<const int32_t*>(ws + W.cta_items);
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
