// attn.cu -- split-context decode attention with folded query heads.
//
// "Core ML Decode Optimization: Removing the 1.9 GiB Per-Token Copy Caused by
// GQA repeat_kv", section 3 ("Fold Q Instead of Expanding KV"): the G query
// rows that share a KV head are handled together as a [G, D] block, so each K
// and V row is read from HBM once and used for all G rows. No replica of K or
// V is made. Scale, mask and softmax act per row and along the context axis.
// prob @ V acts per row. So the context can be split across CTAs and merged
// with a log-sum-exp combine.
//
// "Quest: Query-Aware Sparsity ..." (review), flowchart: the sparse variant
// reads only the K/V rows of the selected pages. It is the same kernel with
// the tile rows taken from a page list instead of a contiguous range.
//
// Kernel shape (one persistent CTA per resident slot, one launch per call):
//  - work tiles: 128 consecutive tokens (dense) or 128 / max(S, 16) selected
//    pages of S tokens (sparse) of one (sequence, KV head) unit. The tiles of all units
//    are split into equal contiguous ranges, one per CTA (balanced split).
//  - warp 8 (producer): TMA tile loads of K and V (both 128-byte swizzled;
//    the E4M3 cache's byte rows 64- or 128-byte swizzled) into a shared-memory
//    ring of 2-6 stages, with mbarrier completion.
//  - warps 0-7 (consumers): fp16 stages: warp w owns 16 tokens of each
//    stage. Low-bit stages: warps 0-3 take the even stages, 4-7 the odd ones
//    (an even ring, so a stage always has the same consumers), and a warp
//    owns 32 tokens of its stages (two 16-token sub-tiles whose MMA chains
//    overlap). Either way a warp runs both products on the tensor cores (MmaAttn:
//    S^T = K Q^T and O^T += V^T P^T with mma.sync m16n8k16, the G folded rows
//    on the N = 8 side), with the online softmax in the log2 domain on the
//    S^T fragments.
//  - at the end of each unit segment the 8 warp states merge in shared
//    memory. A segment that covers its whole unit writes the fp16 output. A
//    segment cut by a range boundary writes an fp32 partial (m, l, acc) and
//    bumps the unit's arrival counter; the CTA that brings the counter to the
//    unit's number of parts merges all of them (log-sum-exp) and writes the
//    output, then sets the counter back to zero for the next call.
#include <math.h>

#include "attn_mma.cuh"
#include "internal.h"

namespace gqaq {

// KV: the cache format. 0 = fp16; 1 = E4M3 codes (one byte per channel:
// half the stage bytes, so up to six stages); 2 = INT4 levels (half a byte
// per channel) with one fp32 scale per token row (up to eight stages).
template <int D, int G, int KV = 0>
struct AttnCfg : TileCfg<D, G> {
    using T = TileCfg<D, G>;
    static constexpr int THREADS = (T::NCW + 1) * 32;
    static constexpr int MISC = 256;
    static constexpr int FIXED = T::QBYTES + T::MERGE + T::PBYTES + MISC;
    static constexpr int KBYTES = KV == 1 ? T::TILE * D : KV == 2 ? T::TILE * D / 2 + T::TILE * 4 : T::KBYTES;
    static constexpr int STAGE = KV != 0 ? 2 * KBYTES : T::STAGE;
    // Low-bit tiles: the deepest even ring of at most six (E4M3) or eight
    // (INT4) stages that fits (two CTAs per SM at D = 64, one at D = 128: at
    // D = 128 two CTAs would leave E4M3 a two-stage ring, measured slower).
    static constexpr int LIMIT8 = (D == 64 ? 112 : 225) * 1024 - FIXED - 1024;
    static constexpr int MAXST = KV == 2 ? 8 : 6;
    static constexpr int NSTAGE8 = (LIMIT8 / STAGE < MAXST ? LIMIT8 / STAGE : MAXST) & ~1;
    static constexpr int NSTAGE = KV != 0 ? NSTAGE8 : ((3 * STAGE + FIXED + 1024 <= 225 * 1024) ? 3 : 2);
    // Low-bit variants: warps 0-3 consume the even stages and warps 4-7 the
    // odd ones, 32 tokens per warp. A stage must then always belong to the
    // same group (an even ring), or a group that skips one of a stage's phases
    // could pass its parity wait a phase early.
    static constexpr bool ALT = KV != 0;
    static_assert(!ALT || NSTAGE % 2 == 0, "alternating warp groups need an even ring");
    static constexpr int SMEM = 1024 + NSTAGE * STAGE + FIXED;
    static constexpr int MIN_BLOCKS = (2 * (SMEM + 1024) <= 228 * 1024) ? 2 : 1;
    static_assert(NSTAGE >= 2, "at least a double-buffered ring");
    static_assert(2 * NSTAGE * 8 + 128 <= MISC, "mbarriers and schedule fit the misc region");
};

constexpr int kMinTilesPerCta = 4;

struct AttnParams {
    const __half *q;
    const int *valid_len;
    const int *page_idx;
    __half *out;
    float *part;      // [grid][2][G][D+2]: fp32 (m, l, acc) of split segments
    unsigned *count;  // [B*Hkv]: arrivals at split units; zero between calls
    int *status;
    int B, Hkv, Lmax, kpages, S;
    float scale_log2;  // includes the K scale of an E4M3 cache
    float v_scale;     // E4M3 cache: V scale (1 otherwise)
    uint64_t timeout_ns;
    int test_stall;
    int early_kv;      // dense: first K/V tiles issued before the grid dependency wait
};

// A unit segment of this CTA that was cut by a range boundary (at most the
// first and the last segment of a range).
struct Split {
    int64_t off;  // tile offset of the unit
    int tiles_b, unit, slot, last;
    __half *out;
};

struct Sched {
    int64_t T;         // tiles of all units
    int64_t t_begin, t_end;
    int64_t unit_off;  // tile offset of the first unit in range
    int b, kv, local, tiles_b, len;
    int grid;          // CTAs with work: min(gridDim.x, T)
    int abort;
    int nsplit;
    Split split[2];
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Walk over the unit segments of one CTA's tile range.
struct Walk {
    int b, kv, local, tiles_b, len;
    int64_t off;  // tile offset of unit (b, kv) in the global tile order
    int64_t remaining;
    bool first;
    __device__ __forceinline__ void init(const Sched &s) {
        b = s.b;
        kv = s.kv;
        local = s.local;
        tiles_b = s.tiles_b;
        len = s.len;
        off = s.unit_off;
        remaining = s.t_end - s.t_begin;
        first = true;
    }
    __device__ __forceinline__ int seg_len() const {
        const int64_t r = tiles_b - local;
        return (int)(r < remaining ? r : remaining);
    }
    // Move past a segment of n tiles; returns false when the range is done.
    __device__ __forceinline__ bool next(int n, const int *valid_len, int B, int Hkv, const TileRule &rule) {
        remaining -= n;
        first = false;
        if (remaining <= 0) return false;
        local = 0;
        off += tiles_b;
        if (++kv == Hkv) {
            kv = 0;
            do {
                if (++b >= B) return false;
                const int raw = valid_len[b];
                len = clamp_len(raw, rule.lmax);
                tiles_b = rule.tiles(raw);
            } while (tiles_b == 0);
        }
        return true;
    }
};

// Log-sum-exp merge of the n_parts partials of one split unit, run by the 256
// consumer threads of the CTA that arrived last (up to FEW parts: one round
// trip to L2 per thread; more: weights first, then the weighted sums):
//   out_g = sum_c 2^(m_c - m*) acc_c / sum_c 2^(m_c - m*) l_c,  m* = max_c m_c.
// The partials of CTAs c_lo .. c_lo + n_parts - 1 sit in slot 0, except the
// first CTA's, whose slot is slot_lo. Other CTAs wrote them, so they are read
// from L2 (ld.global.cg), never from a possibly stale L1 line.
template <int D, int G, int FEW>
__device__ __forceinline__ void merge_parts(const float *part, float *wbuf, int64_t c_lo, int n_parts,
                                            int slot_lo, __half *outg, int warp, int lane, int tid, int nthreads) {
    constexpr int W = G * (D + 2);
    if (n_parts <= FEW) {
        // Few parts: every thread loads (m, l, acc) of its elements from all
        // parts at once and merges them itself (one round trip to L2).
        for (int idx = tid; idx < G * D; idx += nthreads) {
            const int g = idx / D, d = idx - (idx / D) * D;
            float2 ml[FEW];
            float a[FEW];
#pragma unroll
            for (int j = 0; j < FEW; ++j) {
                if (j < n_parts) {
                    const float *ps = part + ((c_lo + j) * 2 + (j == 0 ? slot_lo : 0)) * W + g * (D + 2);
                    ml[j] = __ldcg(reinterpret_cast<const float2 *>(ps));
                    a[j] = __ldcg(ps + 2 + d);
                }
            }
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < FEW; ++j)
                if (j < n_parts) mx = fmaxf(mx, ml[j].x);
            float L = 0.f, acc = 0.f;
#pragma unroll
            for (int j = 0; j < FEW; ++j) {
                if (j < n_parts && ml[j].x != -INFINITY) {
                    const float f = fast_exp2(ml[j].x - mx);
                    L += f * ml[j].y;
                    acc += f * a[j];
                }
            }
            outg[idx] = __float2half_rn(L > 0.f ? acc / L : 0.f);
        }
        return;
    }
    if (warp < G) {
        // Warp g: running (max, sum) over its lanes' parts, then a warp merge.
        float mx = -INFINITY, l = 0.f;
        for (int j = lane; j < n_parts; j += 32) {
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(
                part + ((c_lo + j) * 2 + (j == 0 ? slot_lo : 0)) * W + warp * (D + 2)));
            if (ml.x > mx) {
                l = (mx == -INFINITY) ? ml.y : l * fast_exp2(mx - ml.x) + ml.y;
                mx = ml.x;
            } else if (ml.x != -INFINITY) {
                l += ml.y * fast_exp2(ml.x - mx);
            }
            wbuf[j * G + warp] = ml.x;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, mx, o);
            const float lo = __shfl_xor_sync(0xffffffffu, l, o);
            const float mn = fmaxf(mx, mo);
            l = (mn == -INFINITY) ? 0.f
                                  : (mx == -INFINITY ? 0.f : l * fast_exp2(mx - mn)) +
                                        (mo == -INFINITY ? 0.f : lo * fast_exp2(mo - mn));
            mx = mn;
        }
        __syncwarp();
        for (int j = lane; j < n_parts; j += 32) {
            const float m = wbuf[j * G + warp];
            wbuf[j * G + warp] = (m == -INFINITY) ? 0.f : fast_exp2(m - mx);
        }
        if (lane == 0) wbuf[n_parts * G + warp] = l;
    }
    named_bar_sync(1, nthreads);
    for (int idx = tid; idx < G * D; idx += nthreads) {
        const int g = idx / D, d = idx - (idx / D) * D;
        const float *pe = part + g * (D + 2) + 2 + d;
        float acc = wbuf[g] * __ldcg(pe + (c_lo * 2 + slot_lo) * W);
#pragma unroll 16
        for (int j = 1; j < n_parts; ++j) acc += wbuf[j * G + g] * __ldcg(pe + (c_lo + j) * 2 * W);
        const float L = wbuf[n_parts * G + g];
        outg[idx] = __float2half_rn(L > 0.f ? acc / L : 0.f);
    }
}

// ksmap / vsmap: the INT4 variant's per-token scale rows (unused otherwise).
template <int D, int G, bool SPARSE, int KV = 0>
__global__ void __launch_bounds__(AttnCfg<D, G, KV>::THREADS, AttnCfg<D, G, KV>::MIN_BLOCKS)
    attn_partial_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ CUtensorMap ksmap, const __grid_constant__ CUtensorMap vsmap,
                        const AttnParams p) {
    using C = AttnCfg<D, G, KV>;
    constexpr bool KV8 = KV == 1, KV4 = KV == 2;
    static_assert(!(SPARSE && KV4), "the 4-bit variant is dense");
    constexpr int NCT = C::NCW * 32;  // consumer threads
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stages = smem;
    __half *q_s = reinterpret_cast<__half *>(stages + C::NSTAGE * C::STAGE);
    float *merge = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(q_s) + C::QBYTES);
    float *pbuf = merge + C::NCW * G * (D + 2);
    uint64_t *full = reinterpret_cast<uint64_t *>(pbuf + C::NCW * C::SUB * G);
    uint64_t *empty = full + C::NSTAGE;
    Sched *sched = reinterpret_cast<Sched *>(empty + C::NSTAGE);
    volatile int *abort_flag = &sched->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int Hq = p.Hkv * G;

    // Nothing above the dependency wait reads what an earlier kernel writes.
    if (warp == C::NCW && lane == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), C::ALT ? C::NCW / 2 : C::NCW);  // the warps that consume a stage
        }
        fence_mbar_init();
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        if (KV4) {
            prefetch_tensormap(&ksmap);
            prefetch_tensormap(&vsmap);
        }
    }
    TileRule rule;
    rule.sparse = SPARSE ? 1 : 0;
    rule.lmax = p.Lmax;
    rule.page_size = p.S;
    rule.kpages = p.kpages;
    rule.tile_tokens = C::TILE;
    PageSlots slots;
    slots.init(p.S);
    rule.pages_per_tile = slots.ppt;

    // One dense tile (K and V, and INT4's scale rows) into stage s; lane 0 of the producer.
    auto issue_dense = [&](int s, int unit, int row0, int local, uint64_t pol) {
        const uint32_t kdst = smem_u32(stages + s * C::STAGE);
        const uint32_t vdst = kdst + C::KBYTES;
        const uint32_t fb = smem_u32(&full[s]);
        mbar_arrive_expect_tx(fb, (uint32_t)C::STAGE);
        const int y = row0 + local * C::TILE;
        if (KV4) {  // codes, then the tile's 128 scales (row = unit, x = first token)
            constexpr int CODE4 = C::TILE * D / 2;
            tma_load_2d(kdst, &kmap, 0, y, fb, pol);
            tma_load_2d(kdst + CODE4, &ksmap, local * C::TILE, unit, fb, pol);
            tma_load_2d(vdst, &vmap, 0, y, fb, pol);
            tma_load_2d(vdst + CODE4, &vsmap, local * C::TILE, unit, fb, pol);
        } else if (KV8) {
            tma_load_2d(kdst, &kmap, 0, y, fb, pol);
            tma_load_2d(vdst, &vmap, 0, y, fb, pol);
        } else {
#pragma unroll
            for (int kh = 0; kh < C::KH; ++kh) {
                tma_load_2d(kdst + kh * C::KBLK, &kmap, 64 * kh, y, fb, pol);
                tma_load_2d(vdst + kh * C::KBLK, &vmap, 64 * kh, y, fb, pol);
            }
        }
    };
    // The producer warp's schedule: this CTA's slice of the tile order.
    auto schedule = [&]() {
        // Balanced split of the T tiles over min(gridDim.x, ceil(T / 4)) CTAs:
        // every working CTA owns at least one tile, and a small problem keeps
        // about four per CTA (a short pipeline and few parts per split unit
        // are cheaper than one tile per CTA).
        int64_t T, off_b;
        int b;
        locate_tile(p.valid_len, p.B, p.Hkv, rule, 0, T, b, off_b);
        const int64_t want = (T + kMinTilesPerCta - 1) / kMinTilesPerCta;
        const int gp = (want < (int64_t)gridDim.x) ? (int)(want > 0 ? want : 1) : (int)gridDim.x;
        int64_t tb = 0, te = 0;
        if ((int)blockIdx.x < gp) {
            tb = tile_begin(blockIdx.x, T, gp);
            te = tile_begin(blockIdx.x + 1, T, gp);
        }
        if (tb < te && tb != 0) locate_tile(p.valid_len, p.B, p.Hkv, rule, tb, T, b, off_b);
        if (lane == 0) {
            sched->T = T;
            sched->grid = gp;
            sched->t_begin = tb;
            sched->t_end = te;
            sched->abort = 0;
            sched->nsplit = 0;
            if (tb < te) {
                const int raw = p.valid_len[b];
                const int tiles_b = rule.tiles(raw);
                const int rel = (int)(tb - off_b);  // < Hkv * tiles_b
                sched->b = b;
                sched->kv = rel / tiles_b;
                sched->local = rel - (rel / tiles_b) * tiles_b;
                sched->tiles_b = tiles_b;
                sched->len = clamp_len(raw, p.Lmax);
                sched->unit_off = off_b + (int64_t)(rel / tiles_b) * tiles_b;
            }
        }
    };
    // Early K/V (early_kv): the schedule and the first ring-full of tiles of
    // the first segment are issued before the grid dependency wait, so with a
    // programmatic launch they stream while the previous kernel finishes. The
    // caller guarantees that kernel writes neither valid_len nor any cache row
    // but each sequence's last valid one; the tile holding that row (a unit's
    // last) is left to the loop below. The loop skips the tiles issued here:
    // the same tiles, stages and barrier phases.
    const bool early = !SPARSE && p.early_kv != 0 && p.test_stall == 0;
    int n_early = 0;
    if (early && warp == C::NCW) {
        schedule();
        __syncwarp();  // lane 0's schedule is visible to the warp
        if (lane == 0 && sched->t_begin < sched->t_end) {
            Walk w0;
            w0.init(*sched);
            int lim = w0.seg_len();
            lim = lim < C::NSTAGE ? lim : C::NSTAGE;
            if (w0.local + lim > w0.tiles_b - 1) lim = w0.tiles_b - 1 - w0.local;  // not the unit's last tile
            const uint64_t pol0 = l2_policy_evict_first();
            const int unit = w0.b * p.Hkv + w0.kv;
            for (int t = 0; t < lim; ++t) issue_dense(t, unit, unit * p.Lmax, w0.local + t, pol0);
            n_early = lim > 0 ? lim : 0;
        }
    }
    pdl_wait_and_release();
    if (!early && warp == C::NCW) schedule();
    __syncthreads();

    if (warp < C::NCW) {
        // Sequences with no valid token: defined as a zero output. Lengths
        // outside [1, Lmax] raise GQAQ_DEV_BAD_LEN. CTA b % gridDim.x checks b.
        for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
            const int raw = p.valid_len[b];
            if (threadIdx.x == 0 && (raw < 1 || raw > p.Lmax)) raise_flag(p.status, GQAQ_DEV_BAD_LEN);
            if (rule.tiles(raw) == 0) {
                __half *ob = p.out + (int64_t)b * Hq * D;
                for (int e = threadIdx.x; e < Hq * D; e += NCT) ob[e] = __float2half_rn(0.f);
            }
        }
    }
    if (sched->t_begin >= sched->t_end) return;

    if (warp == C::NCW) {
        // ------------------------------------------------------------------
        // Producer warp
        // ------------------------------------------------------------------
        if (p.test_stall) return;  // issue nothing: every consumer wait runs out
        const uint64_t pol = l2_policy_evict_first();
        Walk w;
        w.init(*sched);
        int i = 0;
        bool failed = false;
        do {
            const int n = w.seg_len();
            const int unit = w.b * p.Hkv + w.kv;
            const int row0 = unit * p.Lmax;
            const int P = (w.len + p.S - 1) / p.S;
            const int nsel = P < p.kpages ? P : p.kpages;
            for (int t = 0; t < n; ++t, ++i) {
                const int s = i % C::NSTAGE;
                const uint32_t ph = (uint32_t)(i / C::NSTAGE) & 1u;
                if (i >= C::NSTAGE) {
                    bool ok = true;
                    if (lane == 0) ok = mbar_wait(smem_u32(&empty[s]), ph ^ 1u, p.timeout_ns, abort_flag);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) {
                        failed = true;
                        break;
                    }
                }
                const uint32_t kdst = smem_u32(stages + s * C::STAGE);
                const uint32_t vdst = kdst + C::KBYTES;
                const uint32_t fb = smem_u32(&full[s]);
                const int local = w.local + t;
                if (SPARSE) {
                    const int e = local * slots.ppt + lane;
                    const bool mine = lane < slots.ppt && e < nsel;
                    int page = -1;
                    if (mine) page = p.page_idx[(int64_t)unit * p.kpages + e];
                    const bool ok = mine && page >= 0 && page < P;
                    if (mine && !ok) raise_flag(p.status, GQAQ_DEV_BAD_PAGE);
                    const unsigned m = __ballot_sync(0xffffffffu, ok);
                    constexpr int RB = KV8 ? D : 2 * D;  // bytes of one cached row
                    if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)__popc(m) * (uint32_t)(p.S * RB * 2));
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int pj = __shfl_sync(0xffffffffu, page, j);
                        if (lane == 0 && ((m >> j) & 1u)) {
                            const int y = row0 + pj * p.S;
                            const uint32_t off = (uint32_t)(j * slots.slot * RB);
                            if (KV8) {  // the page's byte rows land where a dense tile's rows would
                                tma_load_2d(kdst + off, &kmap, 0, y, fb, pol);
                                tma_load_2d(vdst + off, &vmap, 0, y, fb, pol);
                            } else {
                                tma_load_3d(kdst + off, &kmap, 0, 0, y, fb, pol);  // page-major K and V
                                tma_load_3d(vdst + off, &vmap, 0, 0, y, fb, pol);
                            }
                        }
                    }
                } else {
                    if (lane == 0 && i >= n_early) {
                        issue_dense(s, unit, row0, local, pol);
                    }
                }
            }
            if (failed) break;
        } while (w.next(w.seg_len(), p.valid_len, p.B, p.Hkv, rule));
        if (failed) {
            // Let every copy already issued land before this CTA may retire.
            if (lane == 0) {
                raise_flag(p.status, GQAQ_DEV_TIMEOUT);
                *abort_flag = 1;
                const int first = i - C::NSTAGE > 0 ? i - C::NSTAGE : 0;
                for (int it = first; it < i; ++it)
                    mbar_wait(smem_u32(&full[it % C::NSTAGE]), (uint32_t)(it / C::NSTAGE) & 1u,
                              p.timeout_ns, nullptr);
            }
            __syncwarp();
        }
        return;
    }

    // ----------------------------------------------------------------------
    // Consumer warps. After a timeout they still walk every segment and keep
    // the arrival counters in step, so the workspace stays reusable.
    // ----------------------------------------------------------------------
    const int tid = threadIdx.x;  // 0..255 among consumers
    // fp16 sparse stages hold K and V page-major; E4M3 page boxes stack into
    // the dense byte-row layout
    using WA = MmaAttn<D, G, SPARSE && KV == 0, KV>;
    WA wa;
    wa.init(warp, lane, smem_u32(pbuf));

    Walk w;
    w.init(*sched);
    int i = 0;
    do {
        const int n = w.seg_len();
        const bool complete = (w.local == 0 && n == w.tiles_b);
        const int slot = w.first ? 0 : 1;
        const int unit = w.b * p.Hkv + w.kv;
        const int len = w.len;
        const int P = (len + p.S - 1) / p.S;
        const int nsel = P < p.kpages ? P : p.kpages;
        const __half *qg = p.q + ((int64_t)w.b * Hq + (int64_t)w.kv * G) * D;
        if (WA::QREG) {
            wa.load_q(qg);
        } else {
            for (int e = tid; e < G * D / 8; e += NCT)
                reinterpret_cast<uint4 *>(q_s)[e] = reinterpret_cast<const uint4 *>(qg)[e];
            named_bar_sync(1, NCT);
        }
        wa.reset();

        for (int t = 0; t < n; ++t, ++i) {
            if (C::ALT && (i & 1) != (warp >> 2)) continue;  // low-bit: warps 0-3 even stages, 4-7 odd
            const int s = i % C::NSTAGE;
            const uint32_t ph = (uint32_t)(i / C::NSTAGE) & 1u;
            bool ok = (*abort_flag == 0);
            if (ok) {
                if (lane == 0) ok = mbar_wait(smem_u32(&full[s]), ph, p.timeout_ns, abort_flag);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok && lane == 0) {
                    raise_flag(p.status, GQAQ_DEV_TIMEOUT);
                    *abort_flag = 1;
                }
            }
            // this warp's rows of the stage: NS sub-tiles of 16 (virtual warps vw)
            constexpr int NS = C::ALT ? 2 : 1;
            const int local = w.local + t;
            int nv[NS];
#pragma unroll
            for (int h = 0; h < NS; ++h) {
                nv[h] = 0;
                const int vw = C::ALT ? 2 * (warp & 3) + h : warp;
                if (SPARSE) {
                    const int e = local * slots.ppt + slots.warp_page(vw);
                    if (e < nsel) {
                        const int page = p.page_idx[(int64_t)unit * p.kpages + e];
                        if (page >= 0 && page < P) nv[h] = slots.warp_rows(vw, page, len);
                    }
                } else {
                    const int rem = len - (local * C::TILE + vw * C::SUB);
                    nv[h] = rem < 0 ? 0 : (rem < C::SUB ? rem : C::SUB);
                }
            }
            int nsum = 0;
#pragma unroll
            for (int h = 0; h < NS; ++h) nsum += nv[h];
            if (ok && nsum > 0) {
                const uint32_t kbase = smem_u32(stages + s * C::STAGE);
                wa.template tile_n<NS>(kbase, kbase + C::KBYTES, C::ALT ? 32 * (warp & 3) : 16 * warp, nv,
                                       p.scale_log2);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }

        // ---- merge the 8 warp states of this segment ----
        wa.store_state(merge);
        named_bar_sync(1, NCT);
        __half *outg = p.out + ((int64_t)w.b * Hq + (int64_t)w.kv * G) * D;
        for (int idx = tid; idx < G * D; idx += NCT) {
            const int g = idx / D, d = idx - (idx / D) * D;
            float mst, ls, as;
            merge_warps<D, G>(merge, g, d, mst, ls, as);
            if (KV8) as *= p.v_scale;
            if (complete) {
                outg[idx] = __float2half_rn(ls > 0.f ? as / ls : 0.f);
            } else {
                float *ps = p.part + (((int64_t)blockIdx.x * 2 + slot) * G + g) * (D + 2);
                ps[2 + d] = as;
                if (d == 0) {
                    ps[0] = mst;
                    ps[1] = ls;
                }
            }
        }
        named_bar_sync(1, NCT);
        if (!complete && tid == 0) {
            // Arrive at the split unit. The barrier above orders every
            // consumer's partial stores before this release; the unit's last
            // arrival acquires all of them. It has c_hi - c_lo + 1 parts
            // (CTAs c_lo..c_hi, all ranges non-empty). Merging waits for the
            // end of the range.
            Split &sp = sched->split[sched->nsplit++];
            sp.off = w.off;
            sp.tiles_b = w.tiles_b;
            sp.unit = unit;
            sp.slot = slot;
            sp.out = outg;
            const int64_t T = sched->T;
            const int gp = sched->grid;
            const int64_t c_lo = tile_owner(w.off, T, gp);
            const int n_parts = (int)(tile_owner(w.off + w.tiles_b - 1, T, gp) - c_lo) + 1;
            const unsigned old = atomic_add_acq_rel_gpu(&p.count[unit], 1u);
            sp.last = (old + 1u == (unsigned)n_parts);
            if (sp.last) p.count[unit] = 0u;
        }
    } while (w.next(w.seg_len(), p.valid_len, p.B, p.Hkv, rule));

    // ---- merge the split units this CTA arrived at last ----
    named_bar_sync(1, NCT);  // thread 0's arrivals are recorded
    const int nsplit = sched->nsplit;
    if (nsplit == 0) return;
    const int64_t T = sched->T;
    const int gp = sched->grid;
    for (int k = 0; k < nsplit; ++k) {
        const Split &sp = sched->split[k];
        if (!sp.last) continue;
        const int64_t c_lo = tile_owner(sp.off, T, gp);
        const int n_parts = (int)(tile_owner(sp.off + sp.tiles_b - 1, T, gp) - c_lo) + 1;
        const int slot_lo = (tile_begin(c_lo, T, gp) == sp.off) ? 0 : 1;
        // up to FEW parts in one round trip (fewer where two CTAs share an SM's registers)
        merge_parts<D, G, (C::MIN_BLOCKS == 2 ? 8 : 16)>(p.part, merge, c_lo, n_parts, slot_lo, sp.out, warp, lane,
                                                          tid, NCT);
        named_bar_sync(1, NCT);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

constexpr int kMaxDevices = 64;

template <int D, int G, bool SPARSE, int KV = 0>
int grid_for(const LaunchCtx &ctx) {
    using C = AttnCfg<D, G, KV>;
    static int occ[kMaxDevices] = {0};
    if (ctx.device < 0 || ctx.device >= kMaxDevices) return -1;
    if (occ[ctx.device] == 0) {
        auto kern = attn_partial_kernel<D, G, SPARSE, KV>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return -1;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::THREADS, C::SMEM) != cudaSuccess || n < 1)
            return -1;
        occ[ctx.device] = n;
    }
    int grid = occ[ctx.device] * ctx.num_sms;
    if (ctx.max_ctas > 0 && ctx.max_ctas < grid) grid = ctx.max_ctas;
    // The merge keeps (parts + 1) * G weights in the merge buffer.
    if (grid > C::NCW * (D + 2) - 1) grid = C::NCW * (D + 2) - 1;
    return grid;
}

// Workspace: the zero region (arrival counters [B*Hkv] u32 at kWsCounters),
// then the partials [grid][2][G][D+2] fp32.
inline size_t count_bytes(const gqaq_dims &dm) { return workspace_zero_bytes(dm); }

template <int D, int G, bool SPARSE, int KV = 0>
int launch_t(const AttnArgs &a, const LaunchCtx &ctx) {
    using C = AttnCfg<D, G, KV>;
    constexpr bool KV8 = KV == 1, KV4 = KV == 2;
    const gqaq_dims &dm = *a.dims;
    int grid = grid_for<D, G, SPARSE, KV>(ctx);
    if (grid < 1) return GQAQ_ERR_CUDA;
    {
        // Launch no more CTAs than the shape's largest tile count can keep at
        // kMinTilesPerCta tiles each (the kernel applies the same rule to the
        // actual count).
        const int ppt = C::TILE / (dm.page_size > C::SUB ? dm.page_size : C::SUB);  // pages per sparse tile
        const int64_t tiles_unit = SPARSE ? ((int64_t)a.kpages + ppt - 1) / ppt
                                          : ((int64_t)dm.max_len + C::TILE - 1) / C::TILE;
        const int64_t tmax = (int64_t)dm.batch * dm.num_kv_heads * tiles_unit;
        const int64_t want = (tmax + kMinTilesPerCta - 1) / kMinTilesPerCta;
        if (want < grid) grid = (int)(want > 0 ? want : 1);
    }
    const size_t cbytes = count_bytes(dm);
    const size_t need = cbytes + (size_t)grid * 2 * G * (D + 2) * sizeof(float);
    if (a.workspace == nullptr || a.workspace_bytes < need) return GQAQ_ERR_WORKSPACE;

    const uint64_t rows = (uint64_t)dm.batch * dm.num_kv_heads * dm.max_len;
    const uint32_t box_rows = SPARSE ? (uint32_t)dm.page_size : (uint32_t)C::TILE;
    CUtensorMap kmap, vmap, ksmap, vsmap;
    // K and V stages share one layout (the tile reads both through it).
    if (KV4) {  // code rows of D/2 bytes, unswizzled; scale rows [units][Lmax] fp32
        const uint64_t units = (uint64_t)dm.batch * dm.num_kv_heads;
        if (!encode_tensor_map_u8(&kmap, a.k_cache, rows, D / 2, box_rows, 0)) return GQAQ_ERR_CUDA;
        if (!encode_tensor_map_u8(&vmap, a.v_cache, rows, D / 2, box_rows, 0)) return GQAQ_ERR_CUDA;
        if (!encode_tensor_map_f32_rows(&ksmap, a.k_scales, units, dm.max_len, C::TILE)) return GQAQ_ERR_CUDA;
        if (!encode_tensor_map_f32_rows(&vsmap, a.v_scales, units, dm.max_len, C::TILE)) return GQAQ_ERR_CUDA;
    } else if (KV8) {  // byte rows: D = 128 rows 128-byte swizzled, D = 64 rows 64-byte swizzled
        if (!encode_tensor_map_u8(&kmap, a.k_cache, rows, D, box_rows, D == 128 ? 128 : 64)) return GQAQ_ERR_CUDA;
        if (!encode_tensor_map_u8(&vmap, a.v_cache, rows, D, box_rows, D == 128 ? 128 : 64)) return GQAQ_ERR_CUDA;
    } else if (SPARSE) {
        if (!encode_tensor_map_kpage(&kmap, a.k_cache, rows, D, box_rows)) return GQAQ_ERR_CUDA;
        if (!encode_tensor_map_kpage(&vmap, a.v_cache, rows, D, box_rows)) return GQAQ_ERR_CUDA;
    } else {
        if (!encode_tensor_map_2d(&kmap, a.k_cache, rows, D, 64, box_rows, true)) return GQAQ_ERR_CUDA;
        if (!encode_tensor_map_2d(&vmap, a.v_cache, rows, D, 64, box_rows, true)) return GQAQ_ERR_CUDA;
    }
    if (!KV4) {
        ksmap = kmap;  // placeholders: only the INT4 variant reads scale maps
        vsmap = vmap;
    }

    AttnParams p;
    p.q = a.q;
    p.valid_len = a.valid_len;
    p.page_idx = a.page_idx;
    p.out = a.out;
    p.count = reinterpret_cast<unsigned *>(reinterpret_cast<uint8_t *>(a.workspace) + kWsCounters);
    p.part = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(a.workspace) + cbytes);
    p.status = ctx.status;
    p.B = dm.batch;
    p.Hkv = dm.num_kv_heads;
    p.Lmax = dm.max_len;
    p.kpages = SPARSE ? a.kpages : 1;
    p.S = SPARSE ? dm.page_size : 16;
    p.scale_log2 = a.scale * (KV8 ? a.k_scale : 1.f) * 1.4426950408889634f;
    p.v_scale = KV8 ? a.v_scale : 1.f;
    p.timeout_ns = ctx.timeout_ns;
    p.test_stall = ctx.test_stall;
    p.early_kv = ctx.dense_early_kv;
    if (launch_kernel(attn_partial_kernel<D, G, SPARSE, KV>, dim3(grid), dim3(C::THREADS), C::SMEM, ctx, 0, kmap,
                      vmap, ksmap, vsmap, p) != cudaSuccess)
        return GQAQ_ERR_CUDA;
    return GQAQ_OK;
}

template <int D, int G>
int dispatch_sparse(const AttnArgs &a, const LaunchCtx &ctx) {
    if (a.kv8) return a.page_idx ? launch_t<D, G, true, 1>(a, ctx) : launch_t<D, G, false, 1>(a, ctx);
    if (a.kv4) return a.page_idx ? GQAQ_ERR_UNSUPPORTED : launch_t<D, G, false, 2>(a, ctx);
    return a.page_idx ? launch_t<D, G, true>(a, ctx) : launch_t<D, G, false>(a, ctx);
}

template <int D>
int dispatch_g(const AttnArgs &a, const LaunchCtx &ctx, int G) {
    switch (G) {
        case 1: return dispatch_sparse<D, 1>(a, ctx);
        case 2: return dispatch_sparse<D, 2>(a, ctx);
        case 4: return dispatch_sparse<D, 4>(a, ctx);
        case 8: return dispatch_sparse<D, 8>(a, ctx);
        default: return GQAQ_ERR_UNSUPPORTED;
    }
}

template <int D, int G>
size_t ws_t(const gqaq_dims &dm, const LaunchCtx &ctx) {
    const int g0 = grid_for<D, G, false>(ctx);
    const int g1 = grid_for<D, G, true>(ctx);
    const int g2 = grid_for<D, G, false, 1>(ctx);
    const int g3 = grid_for<D, G, false, 2>(ctx);
    const int g4 = grid_for<D, G, true, 1>(ctx);
    if (g0 < 1 || g1 < 1 || g2 < 1 || g3 < 1 || g4 < 1) return 0;
    int grid = g0 > g1 ? g0 : g1;
    grid = grid > g2 ? grid : g2;
    grid = grid > g3 ? grid : g3;
    grid = grid > g4 ? grid : g4;
    return count_bytes(dm) + (size_t)grid * 2 * G * (D + 2) * sizeof(float);
}

template <int D>
size_t ws_g(const gqaq_dims &dm, const LaunchCtx &ctx, int G) {
    switch (G) {
        case 1: return ws_t<D, 1>(dm, ctx);
        case 2: return ws_t<D, 2>(dm, ctx);
        case 4: return ws_t<D, 4>(dm, ctx);
        case 8: return ws_t<D, 8>(dm, ctx);
        default: return 0;
    }
}

}  // namespace

int launch_attention(const AttnArgs &a, const LaunchCtx &ctx) {
    const int G = a.dims->num_q_heads / a.dims->num_kv_heads;
    switch (a.dims->head_dim) {
        case 64: return dispatch_g<64>(a, ctx, G);
        case 128: return dispatch_g<128>(a, ctx, G);
        default: return GQAQ_ERR_UNSUPPORTED;
    }
}

size_t attention_workspace_bytes(const gqaq_dims *dims, const LaunchCtx &ctx) {
    const int G = dims->num_q_heads / dims->num_kv_heads;
    switch (dims->head_dim) {
        case 64: return ws_g<64>(*dims, ctx, G);
        case 128: return ws_g<128>(*dims, ctx, G);
        default: return 0;
    }
}

}  // namespace gqaq
