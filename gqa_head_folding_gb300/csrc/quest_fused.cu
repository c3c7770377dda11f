// quest_fused.cu -- one decode step of a Quest layer in a single launch.
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
// GB300 mapping: a thread-block cluster of C CTAs owns one (sequence, KV
// head) unit at a time (persistent clusters loop over units). Per unit:
//  1. the CTA holding the appended token's page writes the new k, v rows and
//     that page's min/max (producer warp, made visible to TMA by a proxy
//     fence); every CTA streams the metadata of its 1/C of the pages with TMA
//     and scores them on the tensor cores into shared-memory keys (U as a dot
//     of [min(q,0); max(q,0)] with [m; M], since m <= M; pages on the MMA's M
//     side, the G query rows on N);
//  2-3. up to 4096 pages, CTA 0 gathers every key (remote stores into its
//     shared memory) and the scoring warps' key ranges, finds the K-th
//     largest with range-narrowing histogram passes over the keys, and writes
//     each CTA its share of the ascending page list (ties to the lower page
//     index); with more pages,
//     the cluster runs four 8-bit radix passes, summing the C per-CTA
//     histograms through distributed shared memory, and each CTA compacts
//     its own selected pages into every CTA's list;
//  4. each CTA attends over 1/C of the selected pages: each consumer warp
//     fetches its own rows with cp.async (a TMA page gather is bound by the
//     TMA unit's per-box time) and runs the tensor-core tile of attn_mma.cuh;
//  5. each CTA pushes its state (m, l, acc) into the rank that owns each
//     slice of the output; after one cluster barrier every rank merges its
//     slice by log-sum-exp from its own shared memory and writes it in fp16.
// No workspace, no second launch. ATTEND mode runs only steps 4-5 on a page
// list given in global memory.
#include <math.h>
#include <string.h>

#include "attn_mma.cuh"
#include "internal.h"
#include "quest_tile.cuh"

namespace gqaq {

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_ctas() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// Whole-cluster barrier: every thread of every CTA arrives (release) and waits
// (acquire). Shared memory of every CTA in the cluster is visible afterwards.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive without release: for a barrier that only says "this CTA is running".
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_dsmem_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// E4M3 helpers: two fp32 values -> two codes (`lo` in the low byte; round to
// nearest even, magnitudes beyond 448 saturated), one code's value, and the
// canonical code of a bound (zero stored as +0).
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2_q(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(r)
        : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float e4m3_val(uint32_t code) {
    const uint32_t h = e4m3x2_to_f16x2(code & 0xffu);
    return __low2float(*reinterpret_cast<const __half2 *>(&h));
}
__device__ __forceinline__ uint32_t e4m3_canonical(uint32_t code) { return (code & 0x7fu) == 0u ? 0u : code; }

enum { FUSED_FULL = 0, FUSED_ATTEND = 1 };

// KV = 0: fp16 cache and fp16 page bounds; KV = 1: E4M3 codes for both (one
// byte per channel, one scale per tensor).
template <int D, int G, int KV = 0>
struct FusedCfg : TileCfg<D, G> {
    using T = TileCfg<D, G>;
    static constexpr bool KV8 = KV == 1;
    static constexpr int THREADS = (T::NCW + 1) * 32;
    static constexpr int RB = KV8 ? D : 2 * D;      // bytes of one cached row
    static constexpr int KREG = T::TILE * RB;       // K part of a stage (V follows)
    static constexpr int STAGE = 2 * KREG;
    static constexpr int MT = 128;                  // pages per metadata tile
    static constexpr int NB = 2 * RB / 128;         // 128-byte column blocks per [m; M] record
    static constexpr int MBLK = MT * 128;
    static_assert(NB * MBLK == STAGE, "a metadata tile fills one ring stage");
    static constexpr int KEYS_MAX = 4096;           // pages one CTA scores per unit
    static constexpr int KSEL_MAX = 1024;           // selected pages per unit
    static constexpr int KEYMERGE = (KEYS_MAX * 4 > T::MERGE) ? KEYS_MAX * 4 : T::MERGE;
    static constexpr int QREGION = T::QBYTES;       // q of the attention tile when it is staged
    // A cluster rank's inbox: for every source rank, (m, l) of the G rows then
    // the accumulators of the rank's slice of the G*D outputs (<= 8 ranks).
    static constexpr int INBOX = (G * D + 16 * G + 8) * 4;
    // misc region, in 4-byte words: hist [0,512), totals [512,768), unused
    // [768,800), counts [800,808), scan scratch [808,832), scalars [832,848),
    // then the full/empty mbarriers (8-byte aligned) at word 848.
    static constexpr int MISC_BARRIER_WORD = 848;
    static constexpr int NSTAGE_CAP = 3;  // more E4M3 stages (half as large) measured no faster
    static constexpr int MISC = MISC_BARRIER_WORD * 4 + 2 * NSTAGE_CAP * 8;  // full, empty
    static constexpr int FIXED = KEYMERGE + QREGION + T::PBYTES + KSEL_MAX * 4 + INBOX + MISC + 1024;
    static constexpr int NSTAGE_FIT = (226 * 1024 - FIXED - 1024) / STAGE;
    static constexpr int NSTAGE = NSTAGE_FIT > NSTAGE_CAP ? NSTAGE_CAP : (NSTAGE_FIT < 2 ? 2 : NSTAGE_FIT);
    static constexpr int SMEM = 1024 + NSTAGE * STAGE + FIXED;
    static_assert(MISC >= MISC_BARRIER_WORD * 4 + 2 * NSTAGE * 8, "misc region holds the mbarriers");
};

struct FusedParams {
    const __half *q;
    const int *valid_len;
    const int *pos;          // FULL: row of the appended token, or null (no append)
    const __half *k_new, *v_new;
    __half *k_cache, *v_cache, *meta;
    float *scores;           // FULL: optional output
    int *page_idx;           // FULL: optional output; ATTEND: input
    __half *out;
    int *status;
    int B, Hkv, Lmax, Pmax, S, kpages;
    float scale_log2;
    uint64_t timeout_ns;
    int early_meta;          // FULL: first metadata tiles of the first unit issued before the grid dependency wait
    float k_inv, v_inv;      // E4M3 cache: appended rows are quantized as fp32(x) * inv
    float v_scale;           // E4M3 cache: V scale (1 for fp16)
    float score_scale;       // E4M3 cache: K scale of the scores output (1 for fp16)
};

template <int D, int G, int MODE, int KV = 0>
__global__ void __launch_bounds__(FusedCfg<D, G, KV>::THREADS, 1)
    quest_fused_kernel(const __grid_constant__ CUtensorMap mmap, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const FusedParams p) {
    using C = FusedCfg<D, G, KV>;
    constexpr bool KV8 = KV == 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem;
    uint8_t *fixed = ring + C::NSTAGE * C::STAGE;
    uint32_t *keys = reinterpret_cast<uint32_t *>(fixed);      // aliased by merge after step 3
    float *merge = reinterpret_cast<float *>(fixed);
    __half *qreg_s = reinterpret_cast<__half *>(fixed + C::KEYMERGE);
    float *pbuf = reinterpret_cast<float *>(fixed + C::KEYMERGE + C::QREGION);
    int *list = reinterpret_cast<int *>(fixed + C::KEYMERGE + C::QREGION + C::PBYTES);
    float *inbox = reinterpret_cast<float *>(list + C::KSEL_MAX);
    int *misc = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(inbox) + C::INBOX);
    int *hist = misc;                     // [2][256] (cluster radix passes)
    uint32_t *krange = reinterpret_cast<uint32_t *>(misc);  // [2][64] gathered unit: per-warp key min / max
    int *tots = misc + 512;               // [256]
    int *cnt = misc + 800;                // [2] this CTA's (> kth, == kth) counts
    int *wsum = misc + 808;               // [2][9] block-scan scratch
    int *sh = misc + 832;                 // [0] bin, [1] remaining, [2] abort, [3] done, [4..5] key range,
                                          // [6..7] this CTA's key range
    uint64_t *full = reinterpret_cast<uint64_t *>(misc + C::MISC_BARRIER_WORD);
    uint64_t *empty = full + C::NSTAGE;
    volatile int *abort_flag = &sh[2];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t crank = cluster_rank();
    const uint32_t nct = cluster_ctas();
    const int lgc = __ffs((int)nct) - 1;  // cluster sizes are powers of two: shares by shifts
    const int cid = (int)(blockIdx.x >> lgc);
    const int ncl = (int)(gridDim.x >> lgc);
    const int Hq = p.Hkv * G;
    const int units = p.B * p.Hkv;
    const bool producer = (warp == C::NCW);

    if (tid == 0) {  // nothing here reads what an earlier kernel writes
        sh[2] = 0;
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), C::NCW);
        }
        fence_mbar_init();
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        if (MODE == FUSED_FULL) prefetch_tensormap(&mmap);
    }
    // Early metadata (early_meta): the producer issues the first unit's first
    // ring-full of metadata tiles before the grid dependency wait, so with a
    // programmatic launch they stream while the previous kernel finishes. The
    // caller guarantees that kernel writes neither valid_len, pos nor any page
    // other than those holding rows pos-1 and pos; tiles from the one holding
    // either on are left to the loop below, after the wait. They are the same
    // tiles, stages and barrier phases the loop would use, so it skips them.
    int n_early = 0;
    if (MODE == FUSED_FULL && p.early_meta) {
        __syncthreads();  // the ring barriers are initialised
        if (producer && lane == 0 && cid < units) {
            const int b0 = cid / p.Hkv;
            const int P0 = (clamp_len(p.valid_len[b0], p.Lmax) + p.S - 1) / p.S;
            const int q0 = (int)(((int64_t)crank * P0) >> lgc);
            const int q1 = (int)(((int64_t)(crank + 1) * P0) >> lgc);
            int lim = (q1 - q0 + C::MT - 1) / C::MT;
            lim = lim < C::NSTAGE ? lim : C::NSTAGE;
            if (p.pos != nullptr) {
                const int pos0 = p.pos[b0];
                if (pos0 >= 0) {
                    const int pa = (pos0 > 0 ? pos0 - 1 : 0) / p.S, pb = pos0 / p.S;  // pages of rows pos-1, pos
                    if (pa >= q0 && pa < q1) lim = min(lim, (pa - q0) / C::MT);
                    if (pb >= q0 && pb < q1) lim = min(lim, (pb - q0) / C::MT);
                }
            }
            const uint64_t pol0 = l2_policy_evict_first();
            for (int t = 0; t < lim; ++t) {
                const uint32_t fb = smem_u32(&full[t]);
                mbar_arrive_expect_tx(fb, (uint32_t)C::STAGE);
#pragma unroll 1
                for (int kb = 0; kb < C::NB; ++kb)
                    tma_load_2d(smem_u32(ring + t * C::STAGE) + kb * C::MBLK, &mmap, 64 * kb, cid * p.Pmax + q0 + t * C::MT, fb, pol0);
            }
            n_early = lim;
        }
    }
    pdl_wait_and_release();
    // The first unit's length (and appended position) are read before the
    // barriers, so their latency overlaps them.
    const int raw_first = cid < p.B * p.Hkv ? p.valid_len[cid / p.Hkv] : 1;
    const int pos_first = (p.pos != nullptr && cid < p.B * p.Hkv) ? p.pos[cid / p.Hkv] : 0;
    __syncthreads();
    // Every CTA of the cluster must be running before any remote access: the
    // start barrier is arrived at here and waited on just before a thread's
    // first remote access or cluster barrier (cluster_ready), so the first
    // metadata loads and q loads are issued meanwhile.
    // No remote access reads anything written before it, so the arrive is
    // relaxed (a release arrive costs a cluster-scope fence here).
    cluster_arrive_relaxed();
    bool cl_pending = true;
    auto cluster_ready = [&]() {
        if (cl_pending) {
            cluster_wait();
            cl_pending = false;
        }
    };

    const uint64_t pol = l2_policy_evict_first();
    // tensor-core tile: fp16 K and V stages page-major and swizzled; E4M3 byte
    // rows in the layout the 8-bit tile decodes
    using WA = MmaAttn<D, G, !KV8, KV>;
    WA wa;
    wa.init(warp, lane, smem_u32(pbuf));
    int it = 0;  // position in the stage ring (same sequence in producer and consumers)

    for (int u = cid; u < units; u += ncl) {
        const int b = u / p.Hkv, kv = u - (u / p.Hkv) * p.Hkv;
        const int raw = (u == cid) ? raw_first : p.valid_len[b];
        if (tid == 0 && crank == 0 && (raw < 1 || raw > p.Lmax)) raise_flag(p.status, GQAQ_DEV_BAD_LEN);
        const int len = clamp_len(raw, p.Lmax);
        const int P = (len + p.S - 1) / p.S;
        const int nsel = P < p.kpages ? P : p.kpages;
        const __half *qg = p.q + ((int64_t)b * Hq + (int64_t)kv * G) * D;

        if (MODE == FUSED_FULL) {
            // ================= 1. append + page scores =================
            // P <= KEYS_MAX: CTA 0 gathers every key (and their range), selects
            // alone from registers and writes each CTA its share of the page list
            // (two cluster barriers in all). Otherwise each CTA keeps its own keys
            // and the radix passes sum histograms over the cluster.
            const bool gather = P <= C::KEYS_MAX;
            const int pr0 = (int)(((int64_t)crank * P) >> lgc);
            const int pr1 = (int)(((int64_t)(crank + 1) * P) >> lgc);
            const int ntile = (pr1 - pr0 + C::MT - 1) / C::MT;
            if (producer) {
                // The appended token's page is written just before the metadata
                // tile that holds it is loaded (usually the last tile of the last
                // CTA), so the other tiles stream meanwhile.
                int papp = -1;  // page of the appended token when this CTA writes it
                if (p.pos != nullptr) {
                    const int pos = (u == cid) ? pos_first : p.pos[b];
                    if (pos < 0 || pos >= p.Lmax) {
                        if (lane == 0 && crank == 0) raise_flag(p.status, GQAQ_DEV_BAD_POS);
                    } else {
                        const int pg = pos / p.S;
                        if ((pg >= pr0 && pg < pr1) || (crank == nct - 1 && pg >= pr1)) papp = pg;
                    }
                }
                auto append = [&]() {
                    constexpr int EPL = D / 32;
                    const int pos = p.pos[b];
                    if constexpr (KV8) {  // codes of the new rows, then the page's bounds (canonical codes)
                        const int64_t row = ((int64_t)u * p.Lmax + pos) * D + lane * EPL;
                        uint8_t *mrow8 = reinterpret_cast<uint8_t *>(p.meta) + ((int64_t)u * p.Pmax + papp) * 2 * D;
                        uint32_t kw = 0, vw = 0;
#pragma unroll
                        for (int e = 0; e < EPL; e += 2) {
                            const float2 kf = __half22float2(*reinterpret_cast<const __half2 *>(p.k_new + (int64_t)u * D + lane * EPL + e));
                            const float2 vf = __half22float2(*reinterpret_cast<const __half2 *>(p.v_new + (int64_t)u * D + lane * EPL + e));
                            kw |= f32x2_to_e4m3x2_q(kf.x * p.k_inv, kf.y * p.k_inv) << (8 * e);
                            vw |= f32x2_to_e4m3x2_q(vf.x * p.v_inv, vf.y * p.v_inv) << (8 * e);
                        }
                        uint8_t *kc = reinterpret_cast<uint8_t *>(p.k_cache) + row;
                        uint8_t *vc = reinterpret_cast<uint8_t *>(p.v_cache) + row;
                        if (EPL == 4) {
                            *reinterpret_cast<uint32_t *>(kc) = kw;
                            *reinterpret_cast<uint32_t *>(vc) = vw;
                        } else {
                            *reinterpret_cast<uint16_t *>(kc) = (uint16_t)kw;
                            *reinterpret_cast<uint16_t *>(vc) = (uint16_t)vw;
                        }
                        const bool fresh8 = (pos % p.S) == 0;
#pragma unroll
                        for (int e = 0; e < EPL; ++e) {
                            const int c = lane * EPL + e;
                            const uint32_t code = (kw >> (8 * e)) & 0xffu;
                            uint32_t mn = e4m3_canonical(code), mx = mn;
                            if (!fresh8) {
                                const uint32_t om = mrow8[c], oM = mrow8[D + c];
                                const float x = e4m3_val(code);
                                mn = x < e4m3_val(om) ? mn : om;
                                mx = x > e4m3_val(oM) ? mx : oM;
                            }
                            mrow8[c] = (uint8_t)mn;
                            mrow8[D + c] = (uint8_t)mx;
                        }
                        fence_proxy_async_global();  // the TMA reads below see these rows
                        __syncwarp();
                        fence_proxy_async_global();
                        return;
                    }
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
                    fence_proxy_async_global();  // the TMA reads below see these rows
                    __syncwarp();
                    fence_proxy_async_global();
                };
                const int tapp = (papp >= pr0 && papp < pr1) ? (papp - pr0) / C::MT : -1;
                for (int t = 0; t < ntile; ++t, ++it) {
                    const int s = it % C::NSTAGE;
                    const uint32_t ph = (uint32_t)(it / C::NSTAGE) & 1u;
                    if (t == tapp) append();
                    if (it >= C::NSTAGE) {
                        bool ok = (*abort_flag == 0);
                        if (ok && lane == 0) ok = mbar_wait(smem_u32(&empty[s]), ph ^ 1u, p.timeout_ns, abort_flag);
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        if (!ok) {
                            if (lane == 0) { raise_flag(p.status, GQAQ_DEV_TIMEOUT); *abort_flag = 1; }
                            continue;  // keep the ring count in step; issue nothing
                        }
                    }
                    if (lane == 0 && *abort_flag == 0 && !(u == cid && t < n_early)) {
                        const uint32_t fb = smem_u32(&full[s]);
                        const uint32_t dst = smem_u32(ring + s * C::STAGE);
                        mbar_arrive_expect_tx(fb, (uint32_t)C::STAGE);
                        const int y = u * p.Pmax + pr0 + t * C::MT;
#pragma unroll
                        for (int kb = 0; kb < C::NB; ++kb) tma_load_2d(dst + kb * C::MBLK, &mmap, 64 * kb, y, fb, pol);
                    }
                    __syncwarp();
                }
                if (papp >= 0 && tapp < 0) append();  // a page past the valid ones: no tile reads it here
            } else {
                // consumer warps: each scores 16 pages of every tile on the tensor
                // cores, S^T[page][g] = [m; M](page) . [min(q_g, 0); max(q_g, 0)], as
                // one m16n8k16 chain over the 2D-wide record (pages on M, the G query
                // rows on N, columns past G zero and masked), fp32 accumulation.
                constexpr int KS = 2 * D / 16;  // k-steps over the [m; M] record
                uint32_t qb[KS][2];             // B fragments: rows k0, k0+1 (+8) of column lane/4
                {
                    const int n = lane >> 2, k0 = 2 * (lane & 3);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            // record channel of this fragment: c < D is the min side. The
                            // E4M3 record is read as whole 16-byte chunks per lane, so its
                            // contraction order is permuted: k-step ks of column pair
                            // lane%4 covers channels (D/2)(lane%4) + 4 ks .. + 3.
                            const int c = KV8 ? (D / 2) * (lane & 3) + 4 * ks + 2 * h : ks * 16 + k0 + 8 * h;
                            uint32_t v = 0u;
                            if (n < G) {
                                const uint32_t pr = *reinterpret_cast<const uint32_t *>(qg + n * D + (c < D ? c : c - D));
                                v = c < D ? hmin0_bits(pr) : hmax0_bits(pr);
                            }
                            qb[ks][h] = v;
                        }
                }
                cluster_ready();  // the key stores below reach CTA 0
                uint32_t kmn = 0xffffffffu, kmx = 0u;  // range of the keys this lane stores (gather)
                for (int t = 0; t < ntile; ++t, ++it) {
                    const int s = it % C::NSTAGE;
                    const uint32_t ph = (uint32_t)(it / C::NSTAGE) & 1u;
                    bool ok = (*abort_flag == 0);
                    if (ok) {
                        if (lane == 0) ok = mbar_wait(smem_u32(&full[s]), ph, p.timeout_ns, abort_flag);
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        if (!ok && lane == 0) { raise_flag(p.status, GQAQ_DEV_TIMEOUT); *abort_flag = 1; }
                    }
                    const uint32_t sbase = smem_u32(ring + s * C::STAGE);
                    const int first = pr0 + t * C::MT + warp * 16;  // this warp's 16 pages
                    if (ok && first < pr1) {                        // warp-uniform
                        float acc[4] = {0.f, 0.f, 0.f, 0.f};
                        if constexpr (KV8) {
                            // A fragments decoded from the code bytes: page rows r and r + 8
                            // of the warp's 16, this lane's D/2 bytes of each record
                            constexpr int NCH = D / 32;  // 16-byte chunks per lane and row
                            const int ra = warp * 16 + (lane >> 2), rb = ra + 8;
                            uint4 xa[NCH], xb[NCH];
#pragma unroll
                            for (int h = 0; h < NCH; ++h) {
                                const int x = (D / 2) * (lane & 3) + 16 * h;  // record byte
                                const uint32_t blk = sbase + (uint32_t)((x >> 7) * C::MBLK);
                                const uint32_t cx = (uint32_t)((x & 127) >> 4);
                                xa[h] = lds128(blk + (uint32_t)(ra * 128) + ((cx ^ (uint32_t)(ra & 7)) << 4));
                                xb[h] = lds128(blk + (uint32_t)(rb * 128) + ((cx ^ (uint32_t)(rb & 7)) << 4));
                            }
#pragma unroll
                            for (int ks = 0; ks < KS; ++ks) {
                                const uint4 &ua = xa[ks >> 2], &ub = xb[ks >> 2];
                                const uint32_t wa = (ks & 3) == 0 ? ua.x : (ks & 3) == 1 ? ua.y : (ks & 3) == 2 ? ua.z : ua.w;
                                const uint32_t wb = (ks & 3) == 0 ? ub.x : (ks & 3) == 1 ? ub.y : (ks & 3) == 2 ? ub.z : ub.w;
                                uint32_t af[4];
                                e4m3x4_to_f16x2x2(wa, af[0], af[2]);
                                e4m3x4_to_f16x2x2(wb, af[1], af[3]);
                                mma_16816(acc, af, qb[ks][0], qb[ks][1]);
                            }
                        } else {
                            const int arow = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);  // ldmatrix row address
                            const uint32_t abase = sbase + (uint32_t)(arow * 128);
#pragma unroll
                            for (int ks = 0; ks < KS; ++ks) {
                                const uint32_t c16 = (uint32_t)((ks & 3) * 2 + (lane >> 4));
                                uint32_t af[4];
                                ldsm_x4(abase + (uint32_t)((ks >> 2) * C::MBLK) + ((c16 ^ (uint32_t)(arow & 7)) << 4), af);
                                mma_16816(acc, af, qb[ks][0], qb[ks][1]);
                            }
                        }
                        // C fragment: rows lane/4 and lane/4 + 8, columns 2*(lane%4) + {0, 1}
                        const int g0 = 2 * (lane & 3);
                        float b0 = fmaxf(g0 < G ? acc[0] : -INFINITY, g0 + 1 < G ? acc[1] : -INFINITY);
                        float b1 = fmaxf(g0 < G ? acc[2] : -INFINITY, g0 + 1 < G ? acc[3] : -INFINITY);
                        b0 = fmaxf(b0, __shfl_xor_sync(0xffffffffu, b0, 1));
                        b1 = fmaxf(b1, __shfl_xor_sync(0xffffffffu, b1, 1));
                        b0 = fmaxf(b0, __shfl_xor_sync(0xffffffffu, b0, 2));
                        b1 = fmaxf(b1, __shfl_xor_sync(0xffffffffu, b1, 2));
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const float best = half ? b1 : b0;
                            const int page = first + (lane >> 2) + 8 * half;
                            if ((lane & 3) == 0 && page < pr1) {
                                const uint32_t key = score_key(best);
                                if (gather) {  // CTA 0 receives every key of the unit
                                    st_dsmem_u32(dsmem_map(smem_u32(keys + page), 0), key);
                                    kmn = key < kmn ? key : kmn;
                                    kmx = key > kmx ? key : kmx;
                                } else {
                                    keys[page - pr0] = key;
                                }
                                if (p.scores != nullptr) p.scores[(int64_t)u * p.Pmax + page] = best * p.score_scale;
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
                }
                if (gather) {  // this warp's key range into CTA 0's slot (every unit, even if empty)
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        kmn = min(kmn, (uint32_t)__shfl_xor_sync(0xffffffffu, kmn, o));
                        kmx = max(kmx, (uint32_t)__shfl_xor_sync(0xffffffffu, kmx, o));
                    }
                    if (lane == 0) {
                        const int slot = (int)crank * C::NCW + warp;
                        st_dsmem_u32(dsmem_map(smem_u32(&krange[slot]), 0), kmn);
                        st_dsmem_u32(dsmem_map(smem_u32(&krange[64 + slot]), 0), kmx);
                    }
                }
            }
            if (gather) {
                cluster_ready();
                cluster_sync_all();  // CTA 0 holds every key of the unit and its range
            } else {
                __syncthreads();
            }

            if (gather) {
                // ============ 2-3. CTA 0: exact top-K of the gathered keys ============
                // Thread t owns the contiguous run of keys [c0, c1) = [t*chunk, ...).
                // The K-th largest key is located by narrowing a key range [lo, hi],
                // starting from the keys' [min, max]: each pass bins the keys inside
                // it by (key - lo) >> shift into at most 2048 bins (histogram in the
                // idle stage ring) and keeps the bin holding the K-th key, until that
                // bin is wholly selected or holds one key value (one pass, usually).
                // Selected: keys above hi plus the first `need_eq` pages (lowest
                // index) with lo <= key <= hi. Entry `pos` of the ascending page list
                // goes to the CTA whose share [r*nsel/C, (r+1)*nsel/C) contains it.
                // This code runs once per unit on one CTA, so its loops are only
                // lightly unrolled (four independent loads in flight): it is short of
                // instruction-cache hits and load latency, not of issue slots.
                if (crank == 0) {
                    constexpr int NBIN = 2048;
                    static_assert(NBIN * 4 <= C::STAGE, "the histogram fits in one ring stage");
                    int *hb = reinterpret_cast<int *>(ring);
                    const int chunk = (P + C::THREADS - 1) / C::THREADS;
                    const int c0 = tid * chunk < P ? tid * chunk : P;
                    const int c1 = c0 + chunk < P ? c0 + chunk : P;
                    uint32_t lo = 0, hi = 0xffffffffu;
                    int need_eq = P;
                    if (P > p.kpages) {
                        // the unit's key range: the scoring warps' slots, reduced per warp
                        const int nslot = (int)nct * C::NCW;  // <= 64
                        lo = 0xffffffffu;
                        hi = 0u;
                        for (int i = lane; i < nslot; i += 32) {
                            lo = min(lo, krange[i]);
                            hi = max(hi, krange[64 + i]);
                        }
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            lo = min(lo, (uint32_t)__shfl_xor_sync(0xffffffffu, lo, o));
                            hi = max(hi, (uint32_t)__shfl_xor_sync(0xffffffffu, hi, o));
                        }
                        int rem = p.kpages;
                        for (int pass = 0; pass < 4 && lo < hi; ++pass) {
                            const uint32_t span = hi - lo;
                            const int bits = 32 - __clz(span);
                            const int shift = bits > 11 ? bits - 11 : 0;
                            for (int i = tid; i < NBIN; i += C::THREADS) hb[i] = 0;
                            __syncthreads();
#pragma unroll 4
                            for (int i = c0; i < c1; ++i) {
                                const uint32_t k = keys[i];
                                if (k >= lo && k <= hi) atomicAdd(&hb[(k - lo) >> shift], 1);
                            }
                            __syncthreads();
                            // block scan from the top bin down: consumer thread t owns the
                            // 8 bins 2047-8t .. 2040-8t
                            int cc[8], sum = 0;
                            if (tid < C::NCW * 32) {
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    cc[e] = hb[NBIN - 1 - 8 * tid - e];
                                    sum += cc[e];
                                }
                            }
                            int incl = sum;
#pragma unroll
                            for (int o = 1; o < 32; o <<= 1) {
                                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                                if (lane >= o) incl += y;
                            }
                            if (lane == 31 && tid < C::NCW * 32) wsum[warp] = incl;
                            __syncthreads();
                            if (tid < C::NCW * 32) {
                                int before = 0;
                                for (int w = 0; w < warp; ++w) before += wsum[w];
                                const int excl = before + incl - sum;
                                if (excl < rem && rem <= excl + sum) {
                                    int cum = excl;
#pragma unroll
                                    for (int e = 0; e < 8; ++e) {
                                        if (cum + cc[e] >= rem) {
                                            sh[0] = NBIN - 1 - 8 * tid - e;
                                            sh[1] = rem - cum;
                                            sh[3] = (cc[e] == rem - cum) ? 1 : 0;
                                            break;
                                        }
                                        cum += cc[e];
                                    }
                                }
                            }
                            __syncthreads();
                            const uint32_t bsel = (uint32_t)sh[0];
                            const uint32_t nlo = lo + (bsel << shift);
                            const uint32_t top = (bsel << shift) + ((1u << shift) - 1u);
                            hi = lo + (top < span ? top : span);
                            lo = nlo;
                            rem = sh[1];
                            const bool done = sh[3] != 0;
                            __syncthreads();  // sh and the histogram are rewritten next
                            if (done) break;
                        }
                        need_eq = rem;
                    }
                    // ---- compaction: positions from a block scan of (above, in range) ----
                    int ngt = 0, neq = 0;
#pragma unroll 4
                    for (int i = c0; i < c1; ++i) {
                        const uint32_t k = keys[i];
                        ngt += k > hi;
                        neq += k >= lo && k <= hi;
                    }
                    int ig = ngt, ie = neq;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int yg = __shfl_up_sync(0xffffffffu, ig, o);
                        const int ye = __shfl_up_sync(0xffffffffu, ie, o);
                        if (lane >= o) { ig += yg; ie += ye; }
                    }
                    // (the last pass ended at a barrier after its reads of wsum)
                    if (lane == 31) { wsum[warp] = ig; wsum[9 + warp] = ie; }
                    __syncthreads();
                    int bg = 0, be = 0;
                    for (int w = 0; w < warp; ++w) { bg += wsum[w]; be += wsum[9 + w]; }
                    int eqr = be + ie - neq;
                    int pos = bg + ig - ngt + (eqr < need_eq ? eqr : need_eq);
                    // The ascending list is built in the histogram's stage first (a short
                    // loop body), then spread over the cluster by one strided loop.
                    int *sel = hb;
#pragma unroll 4
                    for (int i = c0; i < c1; ++i) {
                        const uint32_t k = keys[i];
                        const bool inr = k >= lo && k <= hi;
                        const bool take = k > hi || (inr && eqr < need_eq);
                        eqr += inr;
                        if (take && pos < nsel) sel[pos] = i;
                        pos += take;
                    }
                    __syncthreads();
                    int *prow = p.page_idx != nullptr ? p.page_idx + (int64_t)u * p.kpages : nullptr;
#pragma unroll 1
                    for (int i = tid; i < nsel; i += C::THREADS) {
                        const int pg = sel[i];
                        const uint32_t owner = (uint32_t)((i + 1) * (int)nct - 1) / (uint32_t)nsel;  // share [r*nsel/C, (r+1)*nsel/C)
                        st_dsmem_u32(dsmem_map(smem_u32(&list[i]), owner), (uint32_t)pg);
                        if (prow != nullptr) prow[i] = pg;
                    }
                    if (prow != nullptr)
                        for (int i = nsel + tid; i < p.kpages; i += C::THREADS) prow[i] = -1;
                    fence_proxy_async_smem();  // the histogram's stage is TMA-written again later
                }
                cluster_ready();
                cluster_sync_all();  // every CTA's share of the page list is in its shared memory
            } else {
                // ================= 2. top-K threshold (adaptive range radix) =================
                // The K-th largest key is located by narrowing a key range [lo, hi]:
                // each pass bins the keys inside it by (key - lo) >> shift into at most
                // 256 bins and keeps the bin holding the K-th key. Starting from the
                // keys' own [min, max] spreads them over the bins (few shared-memory
                // atomics collide), and the loop ends once that bin is wholly selected
                // or holds one key value. Selected: keys above hi, plus the first
                // `need_eq` pages (lowest index) with lo <= key <= hi.
                const bool selecting = true;
                const int nk = gather ? P : pr1 - pr0;
                const int pbase = gather ? 0 : pr0;
                const int e0s = (int)(((int64_t)crank * nsel) >> lgc);       // this CTA's share of the list
                const int e1s = (int)(((int64_t)(crank + 1) * nsel) >> lgc);
                uint32_t lo = 0, hi = 0xffffffffu;
                int need_eq = 0;
                if (P > p.kpages && selecting) {
                    // ---- key range: block min/max (then over the cluster) ----
                    uint32_t kmin = 0xffffffffu, kmax = 0u;
                    for (int i = tid; i < nk; i += C::THREADS) {
                        const uint32_t key = keys[i];
                        kmin = key < kmin ? key : kmin;
                        kmax = key > kmax ? key : kmax;
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        kmin = min(kmin, (uint32_t)__shfl_xor_sync(0xffffffffu, kmin, o));
                        kmax = max(kmax, (uint32_t)__shfl_xor_sync(0xffffffffu, kmax, o));
                    }
                    if (lane == 0) { wsum[warp] = (int)kmin; wsum[9 + warp] = (int)kmax; }
                    __syncthreads();
                    if (tid == 0) {
                        uint32_t a = 0xffffffffu, bmax = 0u;
                        for (int w = 0; w < C::NCW + 1; ++w) {
                            a = min(a, (uint32_t)wsum[w]);
                            bmax = max(bmax, (uint32_t)wsum[9 + w]);
                        }
                        sh[6] = (int)a;  // this CTA's key range, read by the cluster below
                        sh[7] = (int)bmax;
                    }
                    if (!gather) {
                        cluster_ready();
                        cluster_sync_all();
                        if (tid == 0) {
                            uint32_t a = 0xffffffffu, bmax = 0u;
                            for (uint32_t r = 0; r < nct; ++r) {
                                a = min(a, ld_dsmem_u32(dsmem_map(smem_u32(&sh[6]), r)));
                                bmax = max(bmax, ld_dsmem_u32(dsmem_map(smem_u32(&sh[7]), r)));
                            }
                            sh[4] = (int)a;
                            sh[5] = (int)bmax;
                        }
                    } else if (tid == 0) {
                        sh[4] = sh[6];
                        sh[5] = sh[7];
                    }
                    __syncthreads();
                    lo = (uint32_t)sh[4];
                    hi = (uint32_t)sh[5];
                    int rem = p.kpages;
                    for (int pass = 0; pass < 6 && lo < hi; ++pass) {
                        const uint32_t span = hi - lo;  // < 2^32
                        const int bits = 32 - __clz(span);
                        const int shift = bits > 8 ? bits - 8 : 0;
                        int *hb = hist + (pass & 1) * 256;
                        for (int i = tid; i < 256; i += C::THREADS) hb[i] = 0;
                        __syncthreads();
                        for (int i = tid; i < nk; i += C::THREADS) {
                            const uint32_t key = keys[i];
                            if (key >= lo && key <= hi) atomicAdd(&hb[(key - lo) >> shift], 1);
                        }
                        const int *src = hb;
                        if (!gather) {
                            cluster_ready();
                            cluster_sync_all();
                            for (int i = tid; i < 256; i += C::THREADS) {
                                int tot = 0;
                                for (uint32_t r = 0; r < nct; ++r) tot += (int)ld_dsmem_u32(dsmem_map(smem_u32(hb + i), r));
                                tots[i] = tot;
                            }
                            src = tots;
                        }
                        __syncthreads();
                        if (warp == 0) {
                            int c[8], sum = 0;
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                c[e] = src[255 - 8 * lane - e];
                                sum += c[e];
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
                                    if (cum + c[e] >= rem) {
                                        sh[0] = 255 - 8 * lane - e;
                                        sh[1] = rem - cum;
                                        sh[3] = (c[e] == rem - cum) ? 1 : 0;
                                        break;
                                    }
                                    cum += c[e];
                                }
                            }
                        }
                        __syncthreads();
                        const uint32_t bsel = (uint32_t)sh[0];
                        const uint32_t nlo = lo + (bsel << shift);
                        const uint32_t top = (bsel << shift) + ((1u << shift) - 1u);  // <= span
                        hi = lo + (top < span ? top : span);
                        lo = nlo;
                        rem = sh[1];
                        const bool done = sh[3] != 0;
                        __syncthreads();
                        if (done) break;
                    }
                    need_eq = rem;
                }

                // ================= 3. compaction into the ascending page list =================
                if (P > p.kpages && selecting) {
                    const int chunk = (nk + C::THREADS - 1) / C::THREADS;
                    const int c0 = tid * chunk < nk ? tid * chunk : nk;
                    const int c1 = c0 + chunk < nk ? c0 + chunk : nk;
                    int ngt = 0, neq = 0;
                    for (int i = c0; i < c1; ++i) {
                        const uint32_t key = keys[i];
                        ngt += key > hi;
                        neq += key >= lo && key <= hi;
                    }
                    int ig = ngt, ie = neq;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int yg = __shfl_up_sync(0xffffffffu, ig, o);
                        const int ye = __shfl_up_sync(0xffffffffu, ie, o);
                        if (lane >= o) { ig += yg; ie += ye; }
                    }
                    if (lane == 31) { wsum[warp] = ig; wsum[9 + warp] = ie; }
                    __syncthreads();
                    int bg = 0, be = 0, tg = 0, te = 0;
                    for (int w = 0; w < C::NCW + 1; ++w) {
                        if (w < warp) { bg += wsum[w]; be += wsum[9 + w]; }
                        tg += wsum[w];
                        te += wsum[9 + w];
                    }
                    int gt_before = 0, eq_before = 0;
                    if (!gather) {
                        if (tid == 0) { cnt[0] = tg; cnt[1] = te; }
                        cluster_ready();
                        cluster_sync_all();
                        for (uint32_t r = 0; r < crank; ++r) {
                            gt_before += (int)ld_dsmem_u32(dsmem_map(smem_u32(&cnt[0]), r));
                            eq_before += (int)ld_dsmem_u32(dsmem_map(smem_u32(&cnt[1]), r));
                        }
                    }
                    int eqr = eq_before + be + ie - neq;             // rank among equal keys
                    int pos = gt_before + bg + ig - ngt + (eqr < need_eq ? eqr : need_eq);
                    for (int i = c0; i < c1; ++i) {
                        const uint32_t key = keys[i];
                        const bool inr = key >= lo && key <= hi;
                        const bool take = key > hi || (inr && eqr < need_eq);
                        eqr += inr;
                        if (take) {
                            const int page = pbase + i;
                            if (pos < p.kpages && pos < C::KSEL_MAX) {
                                if (!gather) {
                                    for (uint32_t r = 0; r < nct; ++r)
                                        st_dsmem_u32(dsmem_map(smem_u32(&list[pos]), r), (uint32_t)page);
                                    if (p.page_idx != nullptr) p.page_idx[(int64_t)u * p.kpages + pos] = page;
                                } else {
                                    if (pos >= e0s && pos < e1s) list[pos] = page;  // this CTA's share
                                    if (p.page_idx != nullptr && crank == 0) p.page_idx[(int64_t)u * p.kpages + pos] = page;
                                }
                            }
                            ++pos;
                        }
                    }
                } else if (P <= p.kpages) {
                    for (int i = tid; i < P && i < C::KSEL_MAX; i += C::THREADS) list[i] = i;
                    if (p.page_idx != nullptr && crank == 0)
                        for (int i = tid; i < P; i += C::THREADS) p.page_idx[(int64_t)u * p.kpages + i] = i;
                }
                if (p.page_idx != nullptr && crank == 0)
                    for (int i = nsel + tid; i < p.kpages; i += C::THREADS) p.page_idx[(int64_t)u * p.kpages + i] = -1;
                cluster_ready();
                cluster_sync_all();  // remote list entries are complete
            }
        }

        // ================= 4. attention over this CTA's share of the pages =================
        const int e0 = (int)(((int64_t)crank * nsel) >> lgc);
        const int e1 = (int)(((int64_t)(crank + 1) * nsel) >> lgc);
        PageSlots slots;
        slots.init(p.S);
        const int ntile4 = (e1 - e0 + slots.ppt - 1) / slots.ppt;
        if (!producer) {
            if (WA::QREG) {
                wa.load_q(qg);
            } else {
                for (int e = tid; e < G * D / 8; e += C::NCW * 32)
                    reinterpret_cast<uint4 *>(qreg_s)[e] = reinterpret_cast<const uint4 *>(qg)[e];
                named_bar_sync(1, C::NCW * 32);
            }
            wa.reset();
            // Each consumer warp fetches its own 16 rows of every tile with
            // 16-byte cp.async copies into its slice of the idle stage ring, up
            // to NSTAGE tiles ahead, K and V both page-major and 128-byte swizzled
            // (the layout the tensor-core tile reads with ldmatrix): a page
            // gather by TMA is bound by the TMA unit's per-box time, the warps'
            // loads are not.
            // One commit group per tile (empty past the end), so
            // wait_group<NSTAGE - 1> always means "tile t has landed".
            auto in_share = [&](int t) { return t < ntile4 && e0 + t * slots.ppt + slots.warp_page(warp) < e1; };
            auto page_of = [&](int t) {
                if (!in_share(t)) return -1;
                const int e = e0 + t * slots.ppt + slots.warp_page(warp);
                return (MODE == FUSED_FULL) ? list[e] : p.page_idx[(int64_t)u * p.kpages + e];
            };
            auto fetch = [&](int t) {
                const int page = page_of(t);
                if (page >= 0 && page < P) {
                    const int nv = slots.warp_rows(warp, page, len);
                    const int64_t tok0 = (int64_t)u * p.Lmax + (int64_t)page * p.S + (16 * warp) % slots.slot;
                    const uint32_t kb = smem_u32(ring + (t % C::NSTAGE) * C::STAGE), vb = kb + C::KREG;
                    if constexpr (KV8) {  // byte rows: 128-byte swizzle at D = 128, 64-byte at D = 64
                        constexpr int CPR = D / 16;
                        const uint8_t *kg = reinterpret_cast<const uint8_t *>(p.k_cache);
                        const uint8_t *vg = reinterpret_cast<const uint8_t *>(p.v_cache);
                        for (int idx = lane; idx < nv * CPR; idx += 32) {
                            const int i = idx / CPR, c = idx - (idx / CPR) * CPR;
                            const int row = 16 * warp + i;
                            const uint32_t off = D == 128 ? (uint32_t)(row * 128 + ((c ^ (row & 7)) << 4))
                                                          : (uint32_t)(row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
                            cp_async16(kb + off, kg + (tok0 + i) * D + c * 16);
                            cp_async16(vb + off, vg + (tok0 + i) * D + c * 16);
                        }
                    } else {
                        constexpr int CPR = D / 8;  // 16-byte chunks per row
                        for (int idx = lane; idx < nv * CPR; idx += 32) {
                            const int i = idx / CPR, c = idx - (idx / CPR) * CPR;
                            const int row = 16 * warp + i;  // stage row
                            const int line = row * C::KH + (c >> 3);
                            cp_async16(kb + (uint32_t)(line * 128 + (((c & 7) ^ (line & 7)) << 4)),
                                       p.k_cache + (tok0 + i) * D + c * 8);
                            cp_async16(vb + (uint32_t)(line * 128 + (((c & 7) ^ (line & 7)) << 4)),
                                       p.v_cache + (tok0 + i) * D + c * 8);
                        }
                    }
                }
                cp_async_commit();
            };
            for (int t = 0; t < C::NSTAGE; ++t) fetch(t);
            for (int t = 0; t < ntile4; ++t) {
                cp_async_wait<C::NSTAGE - 1>();
                __syncwarp();  // every lane's copies of tile t are visible to the warp
                const int page = page_of(t);
                const bool ok = page >= 0 && page < P;
                if (MODE == FUSED_ATTEND && lane == 0 && in_share(t) && !ok) raise_flag(p.status, GQAQ_DEV_BAD_PAGE);
                const int nv = ok ? slots.warp_rows(warp, page, len) : 0;
                const bool live = __shfl_sync(0xffffffffu, *abort_flag == 0, 0);  // warp-uniform
                if (nv > 0 && live) {
                    const uint32_t kbase = smem_u32(ring + (t % C::NSTAGE) * C::STAGE);
                    const int nvs[1] = {nv};
                    wa.template tile_n<1>(kbase, kbase + C::KREG, 16 * warp, nvs, p.scale_log2);
                }
                __syncwarp();  // the slice is free before tile t + NSTAGE lands in it
                fetch(t + C::NSTAGE);
            }
            cp_async_wait<0>();
            fence_proxy_async_smem();  // the ring is TMA-written again by the next unit
            // ---- merge the 8 warp states; push each rank its slice ----
            // Output i of the G*D belongs to rank i / per. Every rank gets this
            // CTA's (m, l) of all G rows and its accumulators of the rank's slice,
            // in the rank's inbox record for this source, so the merge below reads
            // only local shared memory and no rank reads another after it.
            wa.store_state(merge);
            named_bar_sync(1, C::NCW * 32);
            const int per = (G * D + (int)nct - 1) >> lgc;
            const uint32_t mine = smem_u32(inbox + (int)crank * (2 * G + per));
            for (int idx = tid; idx < G * D; idx += C::NCW * 32) {
                const int g = idx / D, d = idx - (idx / D) * D;
                float mst, ls, as;
                merge_warps<D, G>(merge, g, d, mst, ls, as);
                const int r = idx / per;
                st_dsmem_f32(dsmem_map(mine + 4u * (uint32_t)(2 * G + idx - r * per), (uint32_t)r), as);
                if (d == 0)
                    for (uint32_t q = 0; q < nct; ++q) {
                        st_dsmem_f32(dsmem_map(mine + 8u * (uint32_t)g, q), mst);
                        st_dsmem_f32(dsmem_map(mine + 8u * (uint32_t)g + 4u, q), ls);
                    }
            }
        }
        cluster_ready();
        cluster_sync_all();  // every rank's inbox holds the cluster's states of its slice

        // ================= 5. log-sum-exp merge of this rank's slice =================
        {
            const int per = (G * D + (int)nct - 1) >> lgc;
            const int rec = 2 * G + per;
            const int i0 = (int)crank * per;
            const int i1 = i0 + per < G * D ? i0 + per : G * D;
            for (int idx = i0 + tid; idx < i1; idx += C::THREADS) {
                const int g = idx / D, d = idx - (idx / D) * D;
                float mst = -INFINITY;
                for (uint32_t r = 0; r < nct; ++r) mst = fmaxf(mst, inbox[r * rec + 2 * g]);
                float ls = 0.f, as = 0.f;
                for (uint32_t r = 0; r < nct; ++r) {
                    const float mr = inbox[r * rec + 2 * g];
                    if (mr != -INFINITY) {
                        const float f = fast_exp2(mr - mst);
                        ls += f * inbox[r * rec + 2 * g + 1];
                        as += f * inbox[r * rec + 2 * G + idx - i0];
                    }
                }
                p.out[((int64_t)b * Hq + (int64_t)kv * G + g) * D + d] =
                    __float2half_rn(ls > 0.f ? p.v_scale * (as / ls) : 0.f);
            }
        }
        // Before the next unit reuses keys, list and inbox. After the last unit no
        // rank touches another's shared memory, so the ranks retire without it.
        if (u + ncl < units) {
            cluster_ready();
            cluster_sync_all();
        }
    }

    cluster_ready();  // a cluster with no unit still completes the start barrier

    // If a wait gave up, let this CTA's copies in flight land before it retires.
    if (producer && lane == 0 && *abort_flag) {
        const int first = it - C::NSTAGE > 0 ? it - C::NSTAGE : 0;
        for (int k = first; k < it; ++k)
            mbar_wait(smem_u32(&full[k % C::NSTAGE]), (uint32_t)(k / C::NSTAGE) & 1u, p.timeout_ns, nullptr);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {
constexpr int kMaxDev = 64;

template <int D, int G, int MODE, int KV>
int active_clusters(int device, int csize, int *out) {
    using C = FusedCfg<D, G, KV>;
    static int cache[kMaxDev][4] = {};
    static bool attr[kMaxDev] = {};
    const int ci = csize == 1 ? 0 : csize == 2 ? 1 : csize == 4 ? 2 : 3;
    auto kern = quest_fused_kernel<D, G, MODE, KV>;
    if (!attr[device]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return GQAQ_ERR_CUDA;
        attr[device] = true;
    }
    if (cache[device][ci] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(csize * 64, 1, 1);
        cfg.blockDim = dim3(C::THREADS, 1, 1);
        cfg.dynamicSmemBytes = C::SMEM;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = csize;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
        cache[device][ci] = n > 0 ? n : -1;
    }
    *out = cache[device][ci];
    return GQAQ_OK;
}

template <int D, int G, int MODE, int KV>
int launch_fused_t(const FusedArgs &a, const LaunchCtx &ctx) {
    using C = FusedCfg<D, G, KV>;
    const gqaq_dims &dm = *a.dims;
    const int Pmax = (dm.max_len + dm.page_size - 1) / dm.page_size;
    const int units = dm.batch * dm.num_kv_heads;
    if (a.kpages > C::KSEL_MAX) return GQAQ_ERR_UNSUPPORTED;
    if (ctx.device < 0 || ctx.device >= kMaxDev) return GQAQ_ERR_CUDA;
    // cluster size: smallest C minimising ceil(units / clusters) / C, with Pmax / C <= KEYS_MAX
    int best_c = 0, best_n = 0;
    double best_cost = 1e30;
    for (int csize = 1; csize <= 8; csize *= 2) {
        if (MODE == FUSED_FULL && (Pmax + csize - 1) / csize > C::KEYS_MAX) continue;
        if (ctx.cluster_size > 0 && csize != ctx.cluster_size) continue;
        int n = 0;
        if (active_clusters<D, G, MODE, KV>(ctx.device, csize, &n) != GQAQ_OK) return GQAQ_ERR_CUDA;
        if (n <= 0) continue;
        if (ctx.max_ctas > 0) n = n < ctx.max_ctas / csize ? n : (ctx.max_ctas / csize > 0 ? ctx.max_ctas / csize : 1);
        const double cost = (double)((units + n - 1) / n) / csize;
        if (cost < best_cost * 0.999) {
            best_cost = cost;
            best_c = csize;
            best_n = n;
        }
    }
    if (best_c == 0) return GQAQ_ERR_UNSUPPORTED;
    const int nclusters = units < best_n ? units : best_n;

    const uint64_t rows = (uint64_t)dm.batch * dm.num_kv_heads * dm.max_len;
    CUtensorMap mmap, kmap, vmap;
    if (MODE == FUSED_FULL) {
        const uint64_t mrows = (uint64_t)dm.batch * dm.num_kv_heads * Pmax;
        // a bounds record of 2*RB bytes read as RB halves; 128-byte boxes
        if (!encode_tensor_map_2d(&mmap, a.meta, mrows, C::RB, 64, C::MT, true)) return GQAQ_ERR_CUDA;
    } else {
        memset(&mmap, 0, sizeof(mmap));
    }
    if (KV == 1) {  // byte rows
        if (!encode_tensor_map_u8(&kmap, a.k_cache, rows, D, (uint32_t)dm.page_size, 0)) return GQAQ_ERR_CUDA;
        if (!encode_tensor_map_u8(&vmap, a.v_cache, rows, D, (uint32_t)dm.page_size, 0)) return GQAQ_ERR_CUDA;
    } else {
        if (!encode_tensor_map_kpage(&kmap, a.k_cache, rows, D, (uint32_t)dm.page_size)) return GQAQ_ERR_CUDA;
        if (!encode_tensor_map_2d(&vmap, a.v_cache, rows, D, D, (uint32_t)dm.page_size, false)) return GQAQ_ERR_CUDA;
    }

    FusedParams p;
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
    p.B = dm.batch;
    p.Hkv = dm.num_kv_heads;
    p.Lmax = dm.max_len;
    p.Pmax = Pmax;
    p.S = dm.page_size;
    p.kpages = a.kpages;
    p.scale_log2 = a.scale * (KV == 1 ? a.k_scale : 1.f) * 1.4426950408889634f;
    p.timeout_ns = ctx.timeout_ns;
    p.early_meta = ctx.quest_early_meta;
    p.k_inv = KV == 1 ? a.k_inv : 1.f;
    p.v_inv = KV == 1 ? a.v_inv : 1.f;
    p.v_scale = KV == 1 ? a.v_scale : 1.f;
    p.score_scale = KV == 1 ? a.k_scale : 1.f;

    if (launch_kernel(quest_fused_kernel<D, G, MODE, KV>, dim3(nclusters * best_c), dim3(C::THREADS), C::SMEM, ctx, best_c,
                      mmap, kmap, vmap, p) != cudaSuccess)
        return GQAQ_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? GQAQ_OK : GQAQ_ERR_CUDA;
}

template <int D, int MODE, int KV>
int fused_g(const FusedArgs &a, const LaunchCtx &ctx) {
    switch (a.dims->num_q_heads / a.dims->num_kv_heads) {
        case 1: return launch_fused_t<D, 1, MODE, KV>(a, ctx);
        case 2: return launch_fused_t<D, 2, MODE, KV>(a, ctx);
        case 4: return launch_fused_t<D, 4, MODE, KV>(a, ctx);
        case 8: return launch_fused_t<D, 8, MODE, KV>(a, ctx);
        default: return GQAQ_ERR_UNSUPPORTED;
    }
}
template <int D, int KV>
int fused_mode(const FusedArgs &a, const LaunchCtx &ctx) {
    return a.meta == nullptr ? fused_g<D, FUSED_ATTEND, KV>(a, ctx) : fused_g<D, FUSED_FULL, KV>(a, ctx);
}
}  // namespace

int launch_quest_fused(const FusedArgs &a, const LaunchCtx &ctx) {
    switch (a.dims->head_dim) {
        case 64: return a.kv8 ? fused_mode<64, 1>(a, ctx) : fused_mode<64, 0>(a, ctx);
        case 128: return a.kv8 ? fused_mode<128, 1>(a, ctx) : fused_mode<128, 0>(a, ctx);
        default: return GQAQ_ERR_UNSUPPORTED;
    }
}

}  // namespace gqaq
