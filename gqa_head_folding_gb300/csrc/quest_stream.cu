// quest_stream.cu -- one decode step of a Quest layer as one stream of work
// items over the whole GPU.
//
// "Quest: Query-Aware Sparsity for Efficient Long-Context LLM Inference"
// (reviewer's summary), flowchart: score every page from its key min/max,
// keep the top pages, read only their K and V, attend over those tokens. The
// page-score section: the min/max metadata is updated when a key arrives,
// and U(p,q) = sum_i max(q_i m_{p,i}, q_i M_{p,i}). The token-budget section:
// K pages are kept per query (budget K*S tokens). With grouped query heads
// ("Core ML Decode Optimization ...", section 3), one page set serves the G
// query rows that share a KV head, scored by the largest U over those rows.
//
// GB300 mapping. A persistent grid (one CTA per resident slot) takes work
// items in a fixed order from a ticket counter; each CTA's first item is its
// block index. For every (sequence, KV head) unit u:
//   score items  (u, a): metadata tiles [a*MA, (a+1)*MA) of u (128 pages
//       each). The producer writes the appended token (k, v rows and its
//       page's min/max) when its page falls here, streams the tiles with TMA;
//       the consumers score the pages into u's key array. The arrival that
//       completes u's score items queues u's top-K selection on that CTA.
//   select job (u): exact top-K of u's keys (ties to the lower page index),
//       written as u's ascending page list, then a release flag.
//   attend items (u, c): entries [c*ppi, (c+1)*ppi) of u's page list. The
//       producer waits for u's flag, gathers the pages' K/V with TMA; the
//       consumers attend (the shared warp tile of attn_tile.cuh) and store an
//       fp32 partial (m, l, acc). The arrival that completes u's attend
//       items queues u's merge on that CTA.
//   merge job (u): log-sum-exp of u's partials into the fp16 output.
// All score items precede all attend items in the ticket order, so an attend
// item only waits for score work that running CTAs have already claimed:
// progress never depends on which CTAs are resident.
//
// Inside a CTA, warp 8 (producer) owns the ticket, the TMA issue, the
// arrivals (one gpu-scope fence, then relaxed atomics) and queues jobs into
// the same stage ring the data flows through; warps 0-7 (consumers) process
// ring stages in order. Counters, flags and the ticket live in the caller's
// workspace; they are zero between calls and every call leaves them so.
#include <math.h>

#include "attn_tile.cuh"
#include "internal.h"
#include "quest_tile.cuh"

namespace gqaq {
namespace {

__device__ __forceinline__ unsigned ld_acquire_gpu_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu_u32(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ unsigned atom_add_relaxed_gpu(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void st_release_cta_smem(int *p, int v) {
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta_smem(const int *p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}
__device__ __forceinline__ void fence_proxy_async_global_() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

enum { ST_SCORE = 1, ST_ATTEND = 2, ST_SELECT = 3, ST_MERGE = 4, ST_DONE = 5 };
enum { F_FIRST = 1, F_LAST = 2 };

template <int D, int G>
struct StreamCfg : TileCfg<D, G> {
    using T = TileCfg<D, G>;
    static constexpr int THREADS = (T::NCW + 1) * 32;
    static constexpr int NCT = T::NCW * 32;         // consumer threads
    static constexpr int MT = 128;                  // pages per metadata tile
    static constexpr int NB = 2 * D / 64;           // 128-byte column blocks per [m; M] record
    static_assert(NB * MT * 128 == T::STAGE, "a metadata tile fills one ring stage");
    static constexpr int KPT = 32;                  // keys per consumer thread in a selection
    static constexpr int PSEL_MAX = KPT * NCT;      // pages per unit
    static constexpr int QT_BYTES = G * 2 * D * 2;  // [G][2D] fp16 [q_neg | q_pos]
    static constexpr int QA_BYTES = T::QBYTES;      // attention q block when not in registers
    static constexpr int TI = 12;                   // tile-info words per stage
    static constexpr int IQ = 8;                    // producer's records of items in flight
    static constexpr int PB = 16;                   // arrivals per batch
    static constexpr int NST_MAX = 6;
    // misc region (4-byte words): hist [0,512), wsum [512,528), sh [528,544),
    // done counter [544], item records [548, 564), decisions [564, 564 +
    // NST_MAX), tile info [570, 570 + NST_MAX*TI), then the full/empty mbarriers.
    static constexpr int W_HIST = 0, W_WSUM = 512, W_SH = 528, W_DONE = 544, W_IQ = 548, W_DEC = 564;
    static constexpr int W_TINFO = W_DEC + NST_MAX;
    static constexpr int W_BAR = W_TINFO + NST_MAX * TI;  // 642
    static_assert(W_BAR % 2 == 0, "mbarriers are 8-byte aligned");
    static constexpr int MISC = W_BAR * 4 + 2 * NST_MAX * 8;
    static constexpr int FIXED = T::MERGE + QT_BYTES + QA_BYTES + T::PBYTES + MISC;
    // as many ring stages as fit (at most NST_MAX), one CTA per SM
    static constexpr int NSTAGE_FIT = (226 * 1024 - 1024 - FIXED) / T::STAGE;
    static constexpr int NSTAGE = NSTAGE_FIT < NST_MAX ? NSTAGE_FIT : NST_MAX;
    static_assert(NSTAGE >= 2, "ring");
    static constexpr int SMEM = 1024 + NSTAGE * T::STAGE + FIXED;
    static constexpr int MIN_BLOCKS = 1;
};

struct StreamParams {
    const __half *q;
    const int *valid_len;
    const int *pos;  // row of the appended token per sequence, or null
    const __half *k_new, *v_new;
    __half *k_cache, *v_cache, *meta;
    float *scores;   // optional output [U][Pmax]
    int *page_idx;   // optional output [U][kpages]
    __half *out;
    int *status;
    // workspace
    unsigned *ticket;             // [1]
    unsigned *cnt_s, *cnt_a;      // [U] score / attend arrivals
    unsigned *flag;               // [U] page list published
    unsigned *keys;               // [U][Pmax]
    int *list;                    // [U][kpages]
    float *part;                  // [U][nA_att][G][D+2]
    int B, Hkv, Lmax, Pmax, S, kpages;
    int ma;       // metadata tiles per score item
    int n_s;      // score items per unit
    int ppi;      // list entries per attend item (a multiple of 8, so of the pages per stage)
    int n_a;      // attend items per unit
    int n_items;  // U * (n_s + n_a)
    float scale_log2;
    uint64_t timeout_ns;
    int test_stall;
};

// Log-sum-exp merge of n parts [n][G][D+2] (m, l, acc) into outg [G][D]
// by the NCT consumer threads; parts were written by other CTAs (read from
// L2). wbuf holds (n + 1) * G floats for more than 8 parts.
template <int D, int G>
__device__ __forceinline__ void merge_run(const float *parts, int n, float *wbuf, __half *outg, int warp,
                                          int lane, int tid, int nthreads) {
    constexpr int W = G * (D + 2);
    constexpr int FEW = 8;
    if (n == 0) {
        for (int idx = tid; idx < G * D; idx += nthreads) outg[idx] = __float2half_rn(0.f);
        return;
    }
    if (n <= FEW) {
        for (int idx = tid; idx < G * D; idx += nthreads) {
            const int g = idx / D, d = idx - (idx / D) * D;
            float2 ml[FEW];
            float a[FEW];
#pragma unroll
            for (int j = 0; j < FEW; ++j) {
                if (j < n) {
                    const float *ps = parts + j * W + g * (D + 2);
                    ml[j] = __ldcg(reinterpret_cast<const float2 *>(ps));
                    a[j] = __ldcg(ps + 2 + d);
                }
            }
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < FEW; ++j)
                if (j < n) mx = fmaxf(mx, ml[j].x);
            float L = 0.f, acc = 0.f;
#pragma unroll
            for (int j = 0; j < FEW; ++j) {
                if (j < n && ml[j].x != -INFINITY) {
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
        float mx = -INFINITY;
        for (int j = lane; j < n; j += 32) mx = fmaxf(mx, __ldcg(parts + j * W + warp * (D + 2)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float l = 0.f;
        for (int j = lane; j < n; j += 32) {
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(parts + j * W + warp * (D + 2)));
            const float f = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - mx);
            wbuf[j * G + warp] = f;
            l += f * ml.y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) wbuf[n * G + warp] = l;
    }
    named_bar_sync(1, nthreads);
    for (int idx = tid; idx < G * D; idx += nthreads) {
        const int g = idx / D, d = idx - (idx / D) * D;
        const float *pe = parts + g * (D + 2) + 2 + d;
        float acc = 0.f;
#pragma unroll 16
        for (int j = 0; j < n; ++j) acc += wbuf[j * G + g] * __ldcg(pe + j * W);
        const float L = wbuf[n * G + g];
        outg[idx] = __float2half_rn(L > 0.f ? acc / L : 0.f);
    }
    named_bar_sync(1, nthreads);  // wbuf free again
}

template <int D, int G>
__global__ void __launch_bounds__(StreamCfg<D, G>::THREADS, StreamCfg<D, G>::MIN_BLOCKS)
    quest_stream_kernel(const __grid_constant__ CUtensorMap mmap, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const StreamParams p) {
    using C = StreamCfg<D, G>;
    using MS = MetaScorer<D, G, C::MT>;
    constexpr int NCT = C::NCT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem;
    uint8_t *fixed = ring + C::NSTAGE * C::STAGE;
    float *merge = reinterpret_cast<float *>(fixed);
    __half *qt_s = reinterpret_cast<__half *>(fixed + C::MERGE);
    __half *qa_s = reinterpret_cast<__half *>(fixed + C::MERGE + C::QT_BYTES);
    float *pbuf = reinterpret_cast<float *>(fixed + C::MERGE + C::QT_BYTES + C::QA_BYTES);
    int *misc = reinterpret_cast<int *>(fixed + C::MERGE + C::QT_BYTES + C::QA_BYTES + C::PBYTES);
    int *hist = misc + C::W_HIST;
    int *wsum = misc + C::W_WSUM;
    int *sh = misc + C::W_SH;      // [0] bin, [1] remaining, [2] abort, [3] done, [4..5] key range
    int *done_ctr = misc + C::W_DONE;
    int *iq_kind = misc + C::W_IQ;
    int *iq_unit = misc + C::W_IQ + C::IQ;
    int *dec = misc + C::W_DEC;    // [NSTAGE] consumer decision per ring slot
    int *tinfo = misc + C::W_TINFO;
    uint64_t *full = reinterpret_cast<uint64_t *>(misc + C::W_BAR);
    uint64_t *empty = full + C::NSTAGE;
    volatile int *abort_flag = &sh[2];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hq = p.Hkv * G;
    const int U = p.B * p.Hkv;
    const int n_score = U * p.n_s;

    if (warp == C::NCW && lane == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), C::NCW);
            dec[s] = -2;
        }
        sh[2] = 0;
        *done_ctr = 0;
        fence_mbar_init();
        prefetch_tensormap(&mmap);
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    pdl_wait_and_release();
    __syncthreads();

    if (warp == C::NCW) {
        // ======================================================================
        // Producer warp. Lane 0 owns the ring position, the item records and
        // the arrivals; the warp helps with the append and the page lists.
        // ======================================================================
        if (p.test_stall) return;  // issue nothing: every consumer wait runs out
        const uint64_t pol = l2_policy_evict_first();
        int it = 0;          // ring position (lane 0)
        int issued = 0;      // items recorded (lane 0)
        int seen = 0;        // items whose completion was processed (lane 0)
        int npend = 0;       // arrivals not yet sent (lane 0)
        int pk[C::PB], pu[C::PB];
        bool failed = false;

        // Lane 0: wait for a free ring slot; false on timeout.
        auto slot_wait = [&](int &s) -> bool {
            s = it % C::NSTAGE;
            if (it < C::NSTAGE) return true;
            return mbar_wait(smem_u32(&empty[s]), ((uint32_t)(it / C::NSTAGE) & 1u) ^ 1u, p.timeout_ns, abort_flag);
        };
        // Lane 0: queue a job stage (no data) for the consumers.
        auto queue_job = [&](int kind, int u) -> bool {
            int s;
            if (!slot_wait(s)) return false;
            tinfo[s * C::TI + 0] = kind;
            tinfo[s * C::TI + 1] = u;
            mbar_arrive(smem_u32(&full[s]));
            ++it;
            return true;
        };
        // Lane 0: send the pending arrivals. One fence publishes what this CTA
        // wrote; the arrival that completes a unit's items queues its job.
        auto flush = [&]() -> bool {
            if (npend == 0) return true;
            fence_acq_rel_gpu();
            unsigned old[C::PB];
#pragma unroll
            for (int k = 0; k < C::PB; ++k)
                if (k < npend) old[k] = atom_add_relaxed_gpu((pk[k] == ST_SCORE ? p.cnt_s : p.cnt_a) + pu[k], 1u);
            bool any = false;
            bool last[C::PB];
#pragma unroll
            for (int k = 0; k < C::PB; ++k) {
                last[k] = false;
                if (k < npend) {
                    const unsigned target = (unsigned)(pk[k] == ST_SCORE ? p.n_s : p.n_a);
                    last[k] = (old[k] + 1u == target);
                    any |= last[k];
                }
            }
            if (any) fence_acq_rel_gpu();  // acquire every other CTA's part of the unit
            bool ok = true;
#pragma unroll
            for (int k = 0; k < C::PB; ++k) {
                if (k < npend && last[k]) {
                    if (pk[k] == ST_SCORE) {
                        p.cnt_s[pu[k]] = 0u;
                        ok = ok && queue_job(ST_SELECT, pu[k]);
                    } else {
                        p.cnt_a[pu[k]] = 0u;
                        p.flag[pu[k]] = 0u;  // every attend item of the unit has read it
                        ok = ok && queue_job(ST_MERGE, pu[k]);
                    }
                }
            }
            npend = 0;
            return ok;
        };
        auto add_arrival = [&](int kind, int u) -> bool {
            if (npend == C::PB && !flush()) return false;
            pk[npend] = kind;
            pu[npend] = u;
            ++npend;
            return true;
        };
        // Lane 0: collect the items the consumers finished (in issue order).
        auto collect = [&](bool block) -> bool {
            int nd = ld_acquire_cta_smem(done_ctr);
            if (block && nd == seen) {
                const uint64_t t0 = global_timer_ns();
                while ((nd = ld_acquire_cta_smem(done_ctr)) == seen) {
                    if (*abort_flag || global_timer_ns() - t0 >= p.timeout_ns) return false;
                    __nanosleep(64);
                }
            }
            while (seen < nd) {
                if (!add_arrival(iq_kind[seen % C::IQ], iq_unit[seen % C::IQ])) return false;
                ++seen;
            }
            return flush();
        };
        auto record = [&](int kind, int u) -> bool {
            while (issued - seen >= C::IQ)
                if (!collect(true)) return false;
            iq_kind[issued % C::IQ] = kind;
            iq_unit[issued % C::IQ] = u;
            ++issued;
            return true;
        };

        int item = blockIdx.x;
        unsigned tk = 0;
        bool drew = false;
        while (item < p.n_items) {
            if (lane == 0) {
                tk = atom_add_relaxed_gpu(p.ticket, 1u);  // the next item, used at the end of this one
                drew = true;
            }
            const bool is_score = item < n_score;
            const int rel = is_score ? item : item - n_score;
            const int per = is_score ? p.n_s : p.n_a;
            const int u = rel / per, idx = rel - (rel / per) * per;
            const int b = u / p.Hkv, kv = u - (u / p.Hkv) * p.Hkv;
            const int raw = p.valid_len[b];
            const int len = clamp_len(raw, p.Lmax);
            const int P = (len + p.S - 1) / p.S;
            const int nsel = P < p.kpages ? P : p.kpages;
            bool ok = true;
            if (is_score) {
                if (idx == 0 && kv == 0 && lane == 0 && (raw < 1 || raw > p.Lmax)) raise_flag(p.status, GQAQ_DEV_BAD_LEN);
                const int pg0 = idx * p.ma * C::MT;
                if (p.pos != nullptr) {
                    const int pos = p.pos[b];
                    if (pos < 0 || pos >= p.Lmax) {
                        if (idx == 0 && kv == 0 && lane == 0) raise_flag(p.status, GQAQ_DEV_BAD_POS);
                    } else if (pos / p.S / (p.ma * C::MT) == idx) {
                        // Append: k, v row and the page's min/max, made visible to
                        // the TMA reads of this and other CTAs by proxy fences.
                        constexpr int EPL = D / 32;
                        const int papp = pos / p.S;
                        const int64_t row = (int64_t)u * p.Lmax + pos;
                        __half *mrow = p.meta + ((int64_t)u * p.Pmax + papp) * 2 * D;
                        const bool fresh = (pos % p.S) == 0;
#pragma unroll
                        for (int e = 0; e < EPL; ++e) {
                            const int c = lane * EPL + e;
                            const __half kn = p.k_new[(int64_t)u * D + c];
                            p.k_cache[row * D + c] = kn;
                            p.v_cache[row * D + c] = p.v_new[(int64_t)u * D + c];
                            __half mn = kn, mx = kn;
                            if (!fresh) {
                                const __half om = mrow[c], oM = mrow[D + c];
                                const float kf = __half2float(kn);
                                mn = (kf < __half2float(om)) ? kn : om;
                                mx = (kf > __half2float(oM)) ? kn : oM;
                            }
                            mrow[c] = mn;
                            mrow[D + c] = mx;
                        }
                        fence_proxy_async_global_();
                        __syncwarp();
                        fence_proxy_async_global_();
                    }
                }
                int nt = (P - pg0 + C::MT - 1) / C::MT;
                nt = nt < 0 ? 0 : (nt > p.ma ? p.ma : nt);
                if (lane == 0) {
                    if (nt == 0) {
                        ok = add_arrival(ST_SCORE, u);
                    } else {
                        for (int t = 0; t < nt && ok; ++t) {
                            int s;
                            ok = slot_wait(s);
                            if (!ok) break;
                            const int p0 = pg0 + t * C::MT;
                            int *ti = tinfo + s * C::TI;
                            ti[0] = ST_SCORE;
                            ti[1] = u;
                            ti[2] = (t == 0 ? F_FIRST : 0) | (t == nt - 1 ? F_LAST : 0);
                            ti[3] = p0;
                            ti[4] = (P - p0) < C::MT ? (P - p0) : C::MT;
                            const uint32_t fb = smem_u32(&full[s]);
                            const uint32_t dst = smem_u32(ring + s * C::STAGE);
                            mbar_arrive_expect_tx(fb, (uint32_t)C::STAGE);
                            const int y = u * p.Pmax + p0;
#pragma unroll
                            for (int kb = 0; kb < C::NB; ++kb)
                                tma_load_2d(dst + kb * C::MT * 128, &mmap, 64 * kb, y, fb, pol);
                            ++it;
                        }
                        if (ok) ok = record(ST_SCORE, u);
                    }
                }
            } else {
                const int e_lo = idx * p.ppi;
                const int ne = nsel - e_lo < p.ppi ? nsel - e_lo : p.ppi;
                if (ne <= 0) {
                    if (lane == 0) ok = add_arrival(ST_ATTEND, u);
                } else {
                    // Wait until u's page list is published, sending arrivals
                    // meanwhile (this CTA may hold u's last score item itself).
                    if (lane == 0) {
                        const uint64_t t0 = global_timer_ns();
                        while (ld_acquire_gpu_u32(p.flag + u) == 0u) {
                            if (!collect(false) || *abort_flag || global_timer_ns() - t0 >= p.timeout_ns) {
                                ok = false;
                                break;
                            }
                            __nanosleep(128);
                        }
                        if (ok) fence_proxy_async_global_();
                    }
                    __syncwarp();  // the list loads below follow lane 0's acquire
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    PageSlots slots;
                    slots.init(p.S);
                    const int nt = (ne + slots.ppt - 1) / slots.ppt;
                    for (int t = 0; t < nt && ok; ++t) {
                        int s = 0;
                        if (lane == 0) ok = slot_wait(s);
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        s = __shfl_sync(0xffffffffu, s, 0);
                        if (!ok) break;
                        const int e = e_lo + t * slots.ppt + lane;
                        const bool in = lane < slots.ppt && e < e_lo + ne;
                        int page = -1;
                        if (in) page = __ldcg(p.list + (int64_t)u * p.kpages + e);
                        const bool okp = in && page >= 0 && page < P;
                        const unsigned m = __ballot_sync(0xffffffffu, okp);
                        int *ti = tinfo + s * C::TI;
                        {  // valid rows of consumer warp (lane & 7)
                            const int j = slots.warp_page(lane & 7);
                            const int pw = __shfl_sync(0xffffffffu, page, j);
                            if (lane < 8) ti[4 + lane] = ((m >> j) & 1u) ? slots.warp_rows(lane, pw, len) : 0;
                        }
                        if (lane == 0) {
                            ti[0] = ST_ATTEND;
                            ti[1] = u;
                            ti[2] = (t == 0 ? F_FIRST : 0) | (t == nt - 1 ? F_LAST : 0);
                            ti[3] = idx;
                        }
                        __syncwarp();
                        const uint32_t kdst = smem_u32(ring + s * C::STAGE);
                        const uint32_t vdst = kdst + C::KBYTES;
                        const uint32_t fb = smem_u32(&full[s]);
                        if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)__popc(m) * (uint32_t)(p.S * D * 2 * 2));
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int pj = __shfl_sync(0xffffffffu, page, j);
                            if (lane == 0 && ((m >> j) & 1u)) {
                                const int y = u * p.Lmax + pj * p.S;
                                const uint32_t off = (uint32_t)(j * slots.slot * D * 2);
                                tma_load_3d(kdst + off, &kmap, 0, 0, y, fb, pol);  // page-major K
                                tma_load_2d(vdst + off, &vmap, 0, y, fb, pol);
                            }
                        }
                        if (lane == 0) ++it;
                        __syncwarp();
                    }
                    if (lane == 0 && ok) ok = record(ST_ATTEND, u);
                }
            }
            if (lane == 0 && ok) ok = collect(false);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                failed = true;
                break;
            }
            item = (int)gridDim.x + (int)__shfl_sync(0xffffffffu, tk, 0);
        }
        if (lane == 0) {
            // The draw that returned n_items - 1 was the call's last: reset.
            if (!failed && drew && tk == (unsigned)(p.n_items - 1)) *p.ticket = 0u;
            if (!failed) {
                while (seen < issued && !failed) failed = !collect(true);
                if (!failed) failed = !flush();
            }
            int s;
            if (!failed && slot_wait(s)) {
                tinfo[s * C::TI + 0] = ST_DONE;
                mbar_arrive(smem_u32(&full[s]));
                ++it;
            } else {
                raise_flag(p.status, GQAQ_DEV_TIMEOUT);
                *abort_flag = 1;
                // Let every copy already issued land before this CTA may retire.
                const int first = it - C::NSTAGE > 0 ? it - C::NSTAGE : 0;
                for (int k = first; k < it; ++k)
                    mbar_wait(smem_u32(&full[k % C::NSTAGE]), (uint32_t)(k / C::NSTAGE) & 1u, p.timeout_ns, nullptr);
            }
        }
        __syncwarp();
        return;
    }

    // ==========================================================================
    // Consumer warps: ring stages in order. The stages of one item follow one
    // another in the ring, and an item is processed by one inner loop, so its
    // running state is dead outside it.
    // ==========================================================================
    MS ms;
    ms.init(lane);
    int it = 0, ndone = 0;
    int qt_unit = -1;  // unit whose [q_neg | q_pos] sits in qt_s
    // Wait for ring position `it`. Every consumer warp adopts the first
    // outcome recorded for the position, so all of them take the same path
    // through the barriers. False: give up (timeout somewhere in the CTA).
    auto next_stage = [&]() -> bool {
        const int s = it % C::NSTAGE;
        const uint32_t ph = (uint32_t)(it / C::NSTAGE) & 1u;
        int outcome = 0;
        if (lane == 0) {
            const bool mine = mbar_wait(smem_u32(&full[s]), ph, p.timeout_ns, abort_flag);
            const int expect = it >= C::NSTAGE ? 2 * (it - C::NSTAGE) : -2;
            const int old = atomicCAS(&dec[s], expect, 2 * it + (mine ? 0 : 1));
            outcome = (old == expect) ? (mine ? 0 : 1) : (old & 1);
            // Another warp saw the stage land first: it has landed for good.
            if (outcome == 0 && !mine && !mbar_wait(smem_u32(&full[s]), ph, p.timeout_ns, nullptr)) outcome = 1;
            if (outcome != 0) {
                raise_flag(p.status, GQAQ_DEV_TIMEOUT);
                *abort_flag = 1;
            }
        }
        return __shfl_sync(0xffffffffu, outcome, 0) == 0;
    };
    auto release = [&](int s) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        ++it;
    };
    while (next_stage()) {
        int s = it % C::NSTAGE;
        const int *ti = tinfo + s * C::TI;
        const int kind = ti[0];
        if (kind == ST_DONE) break;
        const int u = ti[1];
        const int b = u / p.Hkv, kv = u - (u / p.Hkv) * p.Hkv;
        const __half *qg = p.q + ((int64_t)b * Hq + (int64_t)kv * G) * D;

        if (kind == ST_SCORE) {
            if (qt_unit != u) {
                MS::load_q_smem(qg, qt_s, tid, NCT);
                qt_unit = u;
                named_bar_sync(1, NCT);
            }
            bool ok = true;
            while (true) {
                const int flags = ti[2], p0 = ti[3], np = ti[4];
                const uint32_t sbase = smem_u32(ring + s * C::STAGE);
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    const int pl0 = warp * 16 + pass * 8;
                    if (pl0 >= np) continue;  // warp-uniform
                    const float best = ms.score_qs(sbase, pl0 + ms.jp, qt_s);
                    const int pl = pl0 + ms.jp;
                    if (ms.qq == 0 && pl < np) {
                        const int page = p0 + pl;
                        p.keys[(int64_t)u * p.Pmax + page] = score_key(best);
                        if (p.scores != nullptr) p.scores[(int64_t)u * p.Pmax + page] = best;
                    }
                }
                release(s);
                if (flags & F_LAST) break;
                if (!(ok = next_stage())) break;
                s = it % C::NSTAGE;
                ti = tinfo + s * C::TI;
            }
            if (!ok) break;
            named_bar_sync(1, NCT);  // every key of the item is stored; qt_s may change
            if (tid == 0) st_release_cta_smem(done_ctr, ++ndone);
        } else if (kind == ST_ATTEND) {
            WarpAttn<D, G, true> wa;  // K stages in page-major layout
            wa.init(warp, lane, smem_u32(pbuf));
            if (C::QREG) {
                wa.load_q(qg);
            } else {
                for (int e = tid; e < G * D / 8; e += NCT)
                    reinterpret_cast<uint4 *>(qa_s)[e] = reinterpret_cast<const uint4 *>(qg)[e];
                named_bar_sync(1, NCT);
            }
            wa.reset();
            const int c = ti[3];
            bool ok = true;
            while (true) {
                const int flags = ti[2];
                const int nv = ti[4 + warp];
                if (nv > 0) {
                    const uint32_t kbase = smem_u32(ring + s * C::STAGE);
                    wa.tile(kbase, kbase + C::KBYTES, nv, p.scale_log2, qa_s);
                }
                release(s);
                if (flags & F_LAST) break;
                if (!(ok = next_stage())) break;
                s = it % C::NSTAGE;
                ti = tinfo + s * C::TI;
            }
            if (!ok) break;
            wa.store_state(merge);
            named_bar_sync(1, NCT);
            float *pc = p.part + ((int64_t)u * p.n_a + c) * (G * (D + 2));
            for (int idx = tid; idx < G * D; idx += NCT) {
                const int g = idx / D, d = idx - (idx / D) * D;
                float mst, ls, as;
                merge_warps<D, G>(merge, g, d, mst, ls, as);
                pc[g * (D + 2) + 2 + d] = as;
                if (d == 0) {
                    pc[g * (D + 2)] = mst;
                    pc[g * (D + 2) + 1] = ls;
                }
            }
            named_bar_sync(1, NCT);  // partial stored, merge buffer and qa_s free
            if (tid == 0) st_release_cta_smem(done_ctr, ++ndone);
        } else if (kind == ST_SELECT) {
            release(s);
            // ---- exact top-K of u's keys (ties to the lower page index) ----
            // Thread t holds keys [t*chunk, t*chunk + kc). The K-th largest key
            // is located by narrowing a range [lo, hi]: each pass bins the keys
            // inside it by (key - lo) >> shift into at most 256 bins and keeps
            // the bin holding the K-th key, until that bin is wholly selected
            // or holds one key value. Selected: keys above hi, plus the first
            // need_eq pages (lowest index) with lo <= key <= hi.
            const int len = clamp_len(p.valid_len[b], p.Lmax);
            const int P = (len + p.S - 1) / p.S;
            const int nsel = P < p.kpages ? P : p.kpages;
            const int chunk = (P + NCT - 1) / NCT;
            const int c0 = tid * chunk < P ? tid * chunk : P;
            const int kc = c0 + chunk < P ? chunk : P - c0;
            const unsigned *ku = p.keys + (int64_t)u * p.Pmax;
            uint32_t kr[C::KPT];
#pragma unroll
            for (int e = 0; e < C::KPT; ++e) kr[e] = e < kc ? __ldcg(ku + c0 + e) : 0u;
            uint32_t lo = 0, hi = 0xffffffffu;
            int need_eq = P;
            if (P > p.kpages) {
                uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
                for (int e = 0; e < C::KPT; ++e)
                    if (e < kc) {
                        kmin = kr[e] < kmin ? kr[e] : kmin;
                        kmax = kr[e] > kmax ? kr[e] : kmax;
                    }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    kmin = min(kmin, (uint32_t)__shfl_xor_sync(0xffffffffu, kmin, o));
                    kmax = max(kmax, (uint32_t)__shfl_xor_sync(0xffffffffu, kmax, o));
                }
                if (lane == 0) {
                    wsum[warp] = (int)kmin;
                    wsum[8 + warp] = (int)kmax;
                }
                named_bar_sync(1, NCT);
                lo = 0xffffffffu;
                hi = 0u;
                for (int w = 0; w < C::NCW; ++w) {
                    lo = min(lo, (uint32_t)wsum[w]);
                    hi = max(hi, (uint32_t)wsum[8 + w]);
                }
                int rem = p.kpages;
                for (int pass = 0; pass < 6 && lo < hi; ++pass) {
                    const uint32_t span = hi - lo;
                    const int bits = 32 - __clz(span);
                    const int shift = bits > 8 ? bits - 8 : 0;
                    int *hb = hist + (pass & 1) * 256;
                    for (int i = tid; i < 256; i += NCT) hb[i] = 0;
                    named_bar_sync(1, NCT);
#pragma unroll
                    for (int e = 0; e < C::KPT; ++e)
                        if (e < kc && kr[e] >= lo && kr[e] <= hi) atomicAdd(&hb[(kr[e] - lo) >> shift], 1);
                    named_bar_sync(1, NCT);
                    if (warp == 0) {
                        int cc[8], sum = 0;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            cc[e] = hb[255 - 8 * lane - e];
                            sum += cc[e];
                        }
                        int incl = sum;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const int y = __shfl_up_sync(0xffffffffu, incl, o);
                            if (lane >= o) incl += y;
                        }
                        const int excl = incl - sum;
                        if (excl < rem && rem <= incl) {
                            int cum = excl;
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                if (cum + cc[e] >= rem) {
                                    sh[0] = 255 - 8 * lane - e;
                                    sh[1] = rem - cum;
                                    sh[3] = (cc[e] == rem - cum) ? 1 : 0;
                                    break;
                                }
                                cum += cc[e];
                            }
                        }
                    }
                    named_bar_sync(1, NCT);
                    const uint32_t bsel = (uint32_t)sh[0];
                    const uint32_t nlo = lo + (bsel << shift);
                    const uint32_t top = (bsel << shift) + ((1u << shift) - 1u);
                    hi = lo + (top < span ? top : span);
                    lo = nlo;
                    rem = sh[1];
                    const bool done = sh[3] != 0;
                    named_bar_sync(1, NCT);  // sh and the other histogram are rewritten next
                    if (done) break;
                }
                need_eq = rem;
            }
            // ---- compaction: list positions from a block scan of (above, in range) ----
            int ngt = 0, neq = 0;
#pragma unroll
            for (int e = 0; e < C::KPT; ++e)
                if (e < kc) {
                    ngt += kr[e] > hi;
                    neq += kr[e] >= lo && kr[e] <= hi;
                }
            int ig = ngt, ie = neq;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int yg = __shfl_up_sync(0xffffffffu, ig, o);
                const int ye = __shfl_up_sync(0xffffffffu, ie, o);
                if (lane >= o) {
                    ig += yg;
                    ie += ye;
                }
            }
            named_bar_sync(1, NCT);  // wsum is reused
            if (lane == 31) {
                wsum[warp] = ig;
                wsum[8 + warp] = ie;
            }
            named_bar_sync(1, NCT);
            int bg = 0, be = 0;
            for (int w = 0; w < warp; ++w) {
                bg += wsum[w];
                be += wsum[8 + w];
            }
            int eqr = be + ie - neq;
            int pos = bg + ig - ngt + (eqr < need_eq ? eqr : need_eq);
            int *lrow = p.list + (int64_t)u * p.kpages;
            int *prow = p.page_idx != nullptr ? p.page_idx + (int64_t)u * p.kpages : nullptr;
#pragma unroll
            for (int e = 0; e < C::KPT; ++e) {
                if (e < kc) {
                    const bool inr = kr[e] >= lo && kr[e] <= hi;
                    const bool take = kr[e] > hi || (inr && eqr < need_eq);
                    eqr += inr;
                    if (take) {
                        if (pos < nsel) {
                            lrow[pos] = c0 + e;
                            if (prow != nullptr) prow[pos] = c0 + e;
                        }
                        ++pos;
                    }
                }
            }
            if (prow != nullptr)
                for (int i = nsel + tid; i < p.kpages; i += NCT) prow[i] = -1;
            named_bar_sync(1, NCT);  // the whole list is stored
            // With no page selected no attend item waits, and the unit's
            // last attend arrival may already have cleared the flag.
            if (tid == 0 && nsel > 0) st_release_gpu_u32(p.flag + u, 1u);
        } else if (kind == ST_MERGE) {
            release(s);
            const int len = clamp_len(p.valid_len[b], p.Lmax);
            const int P = (len + p.S - 1) / p.S;
            const int nsel = P < p.kpages ? P : p.kpages;
            const int nparts = (nsel + p.ppi - 1) / p.ppi;
            __half *outg = p.out + ((int64_t)b * Hq + (int64_t)kv * G) * D;
            merge_run<D, G>(p.part + (int64_t)u * p.n_a * (G * (D + 2)), nparts, merge, outg, warp, lane, tid,
                            NCT);
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
constexpr int kMaxDev = 64;

struct Plan {
    int grid, ma, n_s, ppi, n_a;
    size_t zero_bytes, keys_off, list_off, part_off, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <int D, int G>
int grid_of(int device, int num_sms, int max_ctas) {
    using C = StreamCfg<D, G>;
    static int occ[kMaxDev] = {0};
    if (device < 0 || device >= kMaxDev) return -1;
    if (occ[device] == 0) {
        auto kern = quest_stream_kernel<D, G>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return -1;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::THREADS, C::SMEM) != cudaSuccess || n < 1)
            return -1;
        occ[device] = n;
    }
    int grid = occ[device] * num_sms;
    if (max_ctas > 0 && max_ctas < grid) grid = max_ctas;
    return grid;
}

// Item sizes from the shapes: about four score items and six attend items
// per CTA when every sequence is full.
template <int D, int G>
bool make_plan(const gqaq_dims &dm, int kpages, int grid, Plan &pl) {
    using C = StreamCfg<D, G>;
    const int64_t U = (int64_t)dm.batch * dm.num_kv_heads;
    const int Pmax = (dm.max_len + dm.page_size - 1) / dm.page_size;
    if (Pmax > C::PSEL_MAX || grid < 1) return false;
    const int tiles = (Pmax + C::MT - 1) / C::MT;
    int ma = 1;
    while (ma < tiles && U * ((tiles + 2 * ma - 1) / (2 * ma)) >= 4LL * grid) ma *= 2;
    const int nselmax = kpages < Pmax ? kpages : Pmax;
    int ppi = 8;
    while (ppi < 64 && U * ((nselmax + ppi - 1) / ppi) > 6LL * grid) ppi *= 2;
    // the merge keeps (parts + 1) * G weights in the merge buffer
    while ((nselmax + ppi - 1) / ppi > C::NCW * (D + 2) - 1) ppi *= 2;
    pl.grid = grid;
    pl.ma = ma;
    pl.n_s = (tiles + ma - 1) / ma;
    pl.ppi = ppi;
    pl.n_a = (nselmax + ppi - 1) / ppi;
    if (U * (pl.n_s + pl.n_a) > (int64_t)INT32_MAX / 2) return false;
    pl.zero_bytes = workspace_zero_bytes(dm);
    pl.keys_off = pl.zero_bytes;
    pl.list_off = pl.keys_off + align256((size_t)U * Pmax * sizeof(unsigned));
    pl.part_off = pl.list_off + align256((size_t)U * kpages * sizeof(int));
    pl.total = pl.part_off + align256((size_t)U * pl.n_a * G * (D + 2) * sizeof(float));
    return true;
}

template <int D, int G>
int stream_t(const FusedArgs &a, const LaunchCtx &ctx, size_t *need_out) {
    using C = StreamCfg<D, G>;
    const gqaq_dims &dm = *a.dims;
    const int grid = grid_of<D, G>(ctx.device, ctx.num_sms, ctx.max_ctas);
    if (grid < 1) return GQAQ_ERR_CUDA;
    Plan pl;
    if (!make_plan<D, G>(dm, a.kpages, grid, pl)) return GQAQ_ERR_UNSUPPORTED;
    if (need_out != nullptr) {
        *need_out = pl.total;
        return GQAQ_OK;
    }
    if (a.workspace == nullptr || a.workspace_bytes < pl.total) return GQAQ_ERR_WORKSPACE;

    const int U = dm.batch * dm.num_kv_heads;
    const int Pmax = (dm.max_len + dm.page_size - 1) / dm.page_size;
    const uint64_t rows = (uint64_t)U * dm.max_len;
    const uint64_t mrows = (uint64_t)U * Pmax;
    CUtensorMap mmap, kmap, vmap;
    if (!encode_tensor_map_2d(&mmap, a.meta, mrows, 2 * D, 64, C::MT, true)) return GQAQ_ERR_CUDA;
    if (!encode_tensor_map_kpage(&kmap, a.k_cache, rows, D, (uint32_t)dm.page_size)) return GQAQ_ERR_CUDA;
    if (!encode_tensor_map_2d(&vmap, a.v_cache, rows, D, D, (uint32_t)dm.page_size, false)) return GQAQ_ERR_CUDA;

    uint8_t *ws = reinterpret_cast<uint8_t *>(a.workspace);
    StreamParams p;
    p.q = a.q;
    p.valid_len = a.valid_len;
    p.pos = a.pos;
    p.k_new = a.k_new;
    p.v_new = a.v_new;
    p.k_cache = a.k_cache;
    p.v_cache = a.v_cache;
    p.meta = a.meta;
    p.scores = a.scores;
    p.page_idx = a.page_idx;
    p.out = a.out;
    p.status = ctx.status;
    p.ticket = reinterpret_cast<unsigned *>(ws + kWsTicket);
    p.cnt_s = reinterpret_cast<unsigned *>(ws + kWsCounters);
    p.cnt_a = p.cnt_s + U;
    p.flag = p.cnt_a + U;
    p.keys = reinterpret_cast<unsigned *>(ws + pl.keys_off);
    p.list = reinterpret_cast<int *>(ws + pl.list_off);
    p.part = reinterpret_cast<float *>(ws + pl.part_off);
    p.B = dm.batch;
    p.Hkv = dm.num_kv_heads;
    p.Lmax = dm.max_len;
    p.Pmax = Pmax;
    p.S = dm.page_size;
    p.kpages = a.kpages;
    p.ma = pl.ma;
    p.n_s = pl.n_s;
    p.ppi = pl.ppi;
    p.n_a = pl.n_a;
    p.n_items = U * (pl.n_s + pl.n_a);
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.timeout_ns = ctx.timeout_ns;
    p.test_stall = ctx.test_stall;
    if (launch_kernel(quest_stream_kernel<D, G>, dim3(grid), dim3(C::THREADS), C::SMEM, ctx, 0, mmap, kmap, vmap,
                      p) != cudaSuccess)
        return GQAQ_ERR_CUDA;
    return GQAQ_OK;
}

template <int D>
int stream_g(const FusedArgs &a, const LaunchCtx &ctx, size_t *need) {
    switch (a.dims->num_q_heads / a.dims->num_kv_heads) {
        case 1: return stream_t<D, 1>(a, ctx, need);
        case 2: return stream_t<D, 2>(a, ctx, need);
        case 4: return stream_t<D, 4>(a, ctx, need);
        case 8: return stream_t<D, 8>(a, ctx, need);
        default: return GQAQ_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_quest_stream(const FusedArgs &a, const LaunchCtx &ctx) {
    switch (a.dims->head_dim) {
        case 64: return stream_g<64>(a, ctx, nullptr);
        case 128: return stream_g<128>(a, ctx, nullptr);
        default: return GQAQ_ERR_UNSUPPORTED;
    }
}

size_t quest_stream_workspace_bytes(const gqaq_dims *dims, int kpages, const LaunchCtx &ctx) {
    FusedArgs a = {};
    a.dims = dims;
    a.kpages = kpages;
    size_t need = 0;
    int rc = GQAQ_ERR_UNSUPPORTED;
    switch (dims->head_dim) {
        case 64: rc = stream_g<64>(a, ctx, &need); break;
        case 128: rc = stream_g<128>(a, ctx, &need); break;
        default: break;
    }
    return rc == GQAQ_OK ? need : 0;
}

}  // namespace gqaq
