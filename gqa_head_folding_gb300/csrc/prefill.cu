// prefill.cu -- causal attention of a chunk of q_len new tokens per sequence.
//
// "Core ML Decode Optimization ...", section "Prefill Needs Separate Design":
// with q_len > 1 the G query heads of a KV head and the q_len new tokens are
// merged into one row axis (rank 4 kept), and every row keeps its own causal
// mask. Rows of KV head kv of sequence b are rho = g * q_len + t (g outer, as
// the reshape of [G][q_len] gives), so the [R = G * q_len][D] block of q is
// contiguous and each K / V row is read once for all R rows. Row rho (token
// t of the chunk, whose keys sit at cache rows start .. start+q_len-1)
// attends to cache rows 0 .. start + t.
//
// Kernel shape (one launch):
//  - work item = (sequence, KV head, block of 128 rows); a CTA takes one item
//    and one of `splits` equal slices of its 64-token context tiles.
//  - warp 8 (producer): TMA loads of K and V tiles (64 rows, 128-byte
//    swizzled column blocks) into a 4-6 stage ring, mbarrier completion.
//  - warps 0-7 (consumers): warp w owns rows 16w .. 16w+15 of the item and
//    runs S = Q K^T and O += P V on the tensor cores (mma.sync m16n8k16,
//    fp16 in, fp32 accumulate), with an online softmax in the log2 domain.
//    Only tiles that cross a row's causal limit are masked.
//  - with one split a warp writes its rows' fp16 output. Otherwise every
//    split writes fp32 (m, l, acc) partials and bumps the item's arrival
//    counter; the CTA that completes it merges the partials (log-sum-exp),
//    writes the output and resets the counter for the next call.
#include <math.h>

#include "attn_mma.cuh"
#include "internal.h"

namespace gqaq {
namespace {

template <int D>
struct PrefillCfg {
    static constexpr int NCW = 8;                 // consumer warps
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int RB = NCW * 16;           // rows per item
    static constexpr int TT = 64;                 // tokens per stage
    static constexpr int KH = D / 64;             // 128-byte column blocks per row
    static constexpr int KBLK = TT * 128;
    static constexpr int KBYTES = KH * KBLK;      // = TT * D * 2
    static constexpr int STAGE = 2 * KBYTES;
    static constexpr int NSTAGE = D == 128 ? 4 : 6;
    static constexpr int KS = D / 16;             // k-steps of q.k
    static constexpr int HT = TT / 2;             // tokens per softmax step (half a stage)
    static constexpr int NBH = HT / 8;            // 8-token column blocks of S per half
    static constexpr int DB = D / 8;              // 8-channel column blocks of O
    static constexpr int MAXS = kPrefillMaxSplits;
    static constexpr int WBYTES = RB * MAXS * 4;  // merge weights
    static constexpr int MISC = 256;
    static constexpr int SMEM = 1024 + NSTAGE * STAGE + WBYTES + MISC;
    // One CTA per SM: nine warps of a block spread over the four SM sub-
    // partitions cap a thread at 168 registers, two blocks at 96, and the
    // tile wants about 160 (q, O, S and P fragments).
    static constexpr int MIN_BLOCKS = 1;
    static_assert(2 * NSTAGE * 8 + 16 <= MISC, "mbarriers fit the misc region");
};

struct PrefillParams {
    const __half *q;
    __half *out;
    const int *start;
    float *part;      // [item * splits + split]: ml [RB][2], then acc [RB][D]
    unsigned *count;  // [items]: arrivals; zero between calls
    int *status;
    int B, Hkv, Lmax, q_len, R, nrb, splits;
    float scale_log2;
    uint64_t timeout_ns;
    int test_stall;
};

// Address of the 16-byte chunk (row, ch8) of a [kh][row] 128-byte-swizzled stage.
template <int D>
__device__ __forceinline__ uint32_t stage_chunk(uint32_t base, int row, int ch8) {
    const int kh = ch8 >> 3, cc = ch8 & 7;
    return base + (uint32_t)(kh * PrefillCfg<D>::KBLK + row * 128 + ((cc ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(PrefillCfg<D>::THREADS, PrefillCfg<D>::MIN_BLOCKS)
    prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const PrefillParams p) {
    using C = PrefillCfg<D>;
    constexpr int NCT = C::NCW * 32;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stages = smem;
    float *wbuf = reinterpret_cast<float *>(stages + C::NSTAGE * C::STAGE);
    uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(wbuf) + C::WBYTES);
    uint64_t *empty = full + C::NSTAGE;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + C::NSTAGE);
    int *last_flag = reinterpret_cast<int *>(empty + C::NSTAGE) + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (warp == C::NCW && lane == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), C::NCW);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    pdl_wait_and_release();
    __syncthreads();

    // ---- the work item and this CTA's slice of its context tiles ----
    const int item = blockIdx.x / p.splits, split = blockIdx.x - (blockIdx.x / p.splits) * p.splits;
    const int rb = item % p.nrb, unit = item / p.nrb;  // unit = b * Hkv + kv
    const int b = unit / p.Hkv;
    const int rho0 = rb * C::RB;
    const int nrows = (p.R - rho0) < C::RB ? (p.R - rho0) : C::RB;
    const int st = p.start[b];
    const bool good = st >= 0 && st <= p.Lmax - p.q_len;
    if (!good && threadIdx.x == 0 && split == 0 && rb == 0 && unit % p.Hkv == 0) raise_flag(p.status, GQAQ_DEV_BAD_POS);
    // token offsets t = rho mod q_len spanned by the item's rows
    const int t_first = rho0 % p.q_len, t_last = (rho0 + nrows - 1) % p.q_len;
    const bool wraps = nrows >= p.q_len || t_first > t_last;
    const int t_max = wraps ? p.q_len - 1 : t_last, t_min = wraps ? 0 : t_first;
    const int nt = good ? (st + t_max + C::TT) / C::TT : 0;  // tiles up to the item's last row limit
    const int j0 = (int)(((int64_t)split * nt) / p.splits), j1 = (int)(((int64_t)(split + 1) * nt) / p.splits);
    const int kv_end = st + p.q_len;                         // rows >= kv_end hold no chunk data

    if (warp == C::NCW) {
        // ------------------------------------------------------------------
        // Producer warp
        // ------------------------------------------------------------------
        if (p.test_stall || lane != 0) return;
        const uint64_t pol = l2_policy_evict_first();
        const int row0 = unit * p.Lmax;
        int i = 0;
        bool failed = false;
        for (int j = j0; j < j1; ++j, ++i) {
            const int s = i % C::NSTAGE;
            if (i >= C::NSTAGE &&
                !mbar_wait(smem_u32(&empty[s]), ((uint32_t)(i / C::NSTAGE) & 1u) ^ 1u, p.timeout_ns, abort_flag)) {
                failed = true;
                break;
            }
            const uint32_t kdst = smem_u32(stages + s * C::STAGE), vdst = kdst + C::KBYTES;
            const uint32_t fb = smem_u32(&full[s]);
            mbar_arrive_expect_tx(fb, (uint32_t)C::STAGE);
            const int y = row0 + j * C::TT;
#pragma unroll
            for (int kh = 0; kh < C::KH; ++kh) {
                tma_load_2d(kdst + kh * C::KBLK, &kmap, 64 * kh, y, fb, pol);
                tma_load_2d(vdst + kh * C::KBLK, &vmap, 64 * kh, y, fb, pol);
            }
        }
        if (failed) {
            raise_flag(p.status, GQAQ_DEV_TIMEOUT);
            *abort_flag = 1;
            // let every copy already issued land before this CTA may retire
            const int first = i - C::NSTAGE > 0 ? i - C::NSTAGE : 0;
            for (int it = first; it < i; ++it)
                mbar_wait(smem_u32(&full[it % C::NSTAGE]), (uint32_t)(it / C::NSTAGE) & 1u, p.timeout_ns, nullptr);
        }
        return;
    }

    // ----------------------------------------------------------------------
    // Consumer warps
    // ----------------------------------------------------------------------
    const int tid = threadIdx.x;
    const int r = lane >> 2, c = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
    const bool active = warp * 16 < nrows;  // warp-uniform
    const int rl0 = warp * 16 + r, rl1 = rl0 + 8;  // item-local rows of this lane
    const bool live0 = rl0 < nrows, live1 = rl1 < nrows;
    const int lim0 = st + (rho0 + rl0) % p.q_len, lim1 = st + (rho0 + rl1) % p.q_len;
    const __half *qb = p.q + ((int64_t)unit * p.R + rho0) * D;

    uint32_t qa[C::KS][4];  // A fragments of Q (rows r, r+8)
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
        const __half *q0 = qb + (int64_t)rl0 * D + 16 * ks + 2 * c, *q1 = qb + (int64_t)rl1 * D + 16 * ks + 2 * c;
        qa[ks][0] = live0 ? *reinterpret_cast<const uint32_t *>(q0) : 0u;
        qa[ks][1] = live1 ? *reinterpret_cast<const uint32_t *>(q1) : 0u;
        qa[ks][2] = live0 ? *reinterpret_cast<const uint32_t *>(q0 + 8) : 0u;
        qa[ks][3] = live1 ? *reinterpret_cast<const uint32_t *>(q1 + 8) : 0u;
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[C::DB][4];
#pragma unroll
    for (int nb = 0; nb < C::DB; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;

    int i = 0;
    for (int j = j0; j < j1; ++j, ++i) {
        const int s = i % C::NSTAGE;
        bool ok = (*abort_flag == 0);
        if (ok) {
            if (lane == 0) ok = mbar_wait(smem_u32(&full[s]), (uint32_t)(i / C::NSTAGE) & 1u, p.timeout_ns, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok && lane == 0) {
                raise_flag(p.status, GQAQ_DEV_TIMEOUT);
                *abort_flag = 1;
            }
        }
        if (ok && active) {
            const uint32_t kbase = smem_u32(stages + s * C::STAGE), vbase = kbase + C::KBYTES;
            // two 32-token halves per stage: fewer live S / P fragments
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int tok0 = j * C::TT + hf * C::HT, trow = hf * C::HT;  // first token, its stage row
                // ---- S = Q K^T: 16 rows x 32 tokens ----
                float sc[C::NBH][4];
#pragma unroll
                for (int nb = 0; nb < C::NBH; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) {
#pragma unroll
                    for (int pp = 0; pp < C::NBH / 2; ++pp) {
                        uint32_t kf[4];
                        ldsm_x4(stage_chunk<D>(kbase, trow + 16 * pp + (mi >> 1) * 8 + rr, 2 * ks + (mi & 1)), kf);
                        mma_16816(sc[2 * pp], qa[ks], kf[0], kf[1]);
                        mma_16816(sc[2 * pp + 1], qa[ks], kf[2], kf[3]);
                    }
                }
                // ---- causal mask (only where a row limit falls inside), online softmax ----
                const bool need_mask = tok0 + C::HT - 1 > st + t_min;  // uniform over the item
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int nb = 0; nb < C::NBH; ++nb) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tok = tok0 + 8 * nb + 2 * c + e;
                        float x0 = sc[nb][e] * p.scale_log2, x1 = sc[nb][2 + e] * p.scale_log2;
                        if (need_mask) {
                            x0 = tok <= lim0 ? x0 : -INFINITY;
                            x1 = tok <= lim1 ? x1 : -INFINITY;
                        }
                        sc[nb][e] = x0;
                        sc[nb][2 + e] = x1;
                        mx0 = fmaxf(mx0, x0);
                        mx1 = fmaxf(mx1, x1);
                    }
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                // a row with no valid token yet keeps a zero reference (no inf - inf)
                const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
                const float al0 = fast_exp2(m0 - ref0), al1 = fast_exp2(m1 - ref1);
                m0 = mn0;
                m1 = mn1;
                float ps0 = 0.f, ps1 = 0.f;
                uint32_t pa[C::NBH / 2][4];  // A fragments of P, 16 tokens each
#pragma unroll
                for (int nb = 0; nb < C::NBH; ++nb) {
                    const float e0 = fast_exp2(sc[nb][0] - ref0), e1 = fast_exp2(sc[nb][1] - ref0);
                    const float e2 = fast_exp2(sc[nb][2] - ref1), e3 = fast_exp2(sc[nb][3] - ref1);
                    ps0 += e0 + e1;
                    ps1 += e2 + e3;
                    pa[nb >> 1][(nb & 1) * 2 + 0] = pack_half2(e0, e1);
                    pa[nb >> 1][(nb & 1) * 2 + 1] = pack_half2(e2, e3);
                }
                l0 = l0 * al0 + ps0;
                l1 = l1 * al1 + ps1;
                if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                    for (int nb = 0; nb < C::DB; ++nb) {
                        o[nb][0] *= al0;
                        o[nb][1] *= al0;
                        o[nb][2] *= al1;
                        o[nb][3] *= al1;
                    }
                }
                // ---- O += P V ----
                const bool tail = tok0 + C::HT > kv_end;  // rows past the chunk: V may hold anything
#pragma unroll
                for (int kk = 0; kk < C::NBH / 2; ++kk) {
                    uint32_t mk0 = 0xffffffffu, mk1 = 0xffffffffu;
                    if (tail) {
                        const int t0 = tok0 + 16 * kk + 2 * c;
                        mk0 = (t0 < kv_end ? 0x0000ffffu : 0u) | (t0 + 1 < kv_end ? 0xffff0000u : 0u);
                        mk1 = (t0 + 8 < kv_end ? 0x0000ffffu : 0u) | (t0 + 9 < kv_end ? 0xffff0000u : 0u);
                    }
#pragma unroll
                    for (int qq = 0; qq < C::DB / 2; ++qq) {
                        uint32_t vf[4];
                        ldsm_x4_trans(stage_chunk<D>(vbase, trow + 16 * kk + (mi & 1) * 8 + rr, 2 * qq + (mi >> 1)),
                                      vf);
                        if (tail) {
                            vf[0] &= mk0;
                            vf[1] &= mk1;
                            vf[2] &= mk0;
                            vf[3] &= mk1;
                        }
                        mma_16816(o[2 * qq], pa[kk], vf[0], vf[1]);
                        mma_16816(o[2 * qq + 1], pa[kk], vf[2], vf[3]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }

    // ---- rows' sums over the 4 lanes of a row ----
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    __half *ob = p.out + ((int64_t)unit * p.R + rho0) * D;
    if (p.splits == 1) {
        const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
        for (int nb = 0; nb < C::DB; ++nb) {
            if (live0)
                *reinterpret_cast<__half2 *>(ob + (int64_t)rl0 * D + 8 * nb + 2 * c) =
                    __floats2half2_rn(o[nb][0] * inv0, o[nb][1] * inv0);
            if (live1)
                *reinterpret_cast<__half2 *>(ob + (int64_t)rl1 * D + 8 * nb + 2 * c) =
                    __floats2half2_rn(o[nb][2] * inv1, o[nb][3] * inv1);
        }
        return;
    }

    // ---- split: fp32 partial, arrival, and the last arrival's merge ----
    float *pml = p.part + (int64_t)blockIdx.x * C::RB * (D + 2);
    float *pacc = pml + 2 * C::RB;
    if (c == 0) {
        if (live0) reinterpret_cast<float2 *>(pml)[rl0] = make_float2(m0, l0);
        if (live1) reinterpret_cast<float2 *>(pml)[rl1] = make_float2(m1, l1);
    }
#pragma unroll
    for (int nb = 0; nb < C::DB; ++nb) {
        if (live0) *reinterpret_cast<float2 *>(pacc + (int64_t)rl0 * D + 8 * nb + 2 * c) = make_float2(o[nb][0], o[nb][1]);
        if (live1) *reinterpret_cast<float2 *>(pacc + (int64_t)rl1 * D + 8 * nb + 2 * c) = make_float2(o[nb][2], o[nb][3]);
    }
    named_bar_sync(1, NCT);
    if (tid == 0) {
        // The barrier orders every consumer's partial stores before this
        // release; the item's last arrival acquires all of them.
        const unsigned old = atomic_add_acq_rel_gpu(&p.count[item], 1u);
        const int last = old + 1u == (unsigned)p.splits;
        if (last) p.count[item] = 0u;
        *last_flag = last;
    }
    named_bar_sync(1, NCT);
    if (!*last_flag) return;

    // weights per (row, split): 2^(m_s - m*) / sum_s 2^(m_s - m*) l_s
    const float *base = p.part + (int64_t)item * p.splits * C::RB * (D + 2);
    for (int row = tid; row < nrows; row += NCT) {
        float mst = -INFINITY;
        for (int sp = 0; sp < p.splits; ++sp)
            mst = fmaxf(mst, __ldcg(base + (int64_t)sp * C::RB * (D + 2) + 2 * row));
        float L = 0.f;
        for (int sp = 0; sp < p.splits; ++sp) {
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(base + (int64_t)sp * C::RB * (D + 2)) + row);
            const float f = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - mst);
            wbuf[row * C::MAXS + sp] = f;
            L += f * ml.y;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int sp = 0; sp < p.splits; ++sp) wbuf[row * C::MAXS + sp] *= inv;
    }
    named_bar_sync(1, NCT);
    for (int e = tid; e < nrows * (D / 4); e += NCT) {
        const int row = e / (D / 4), d4 = e - (e / (D / 4)) * (D / 4);
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < p.splits; ++sp) {
            const float w = wbuf[row * C::MAXS + sp];
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(base + (int64_t)sp * C::RB * (D + 2) + 2 * C::RB +
                                                                     (int64_t)row * D) + d4);
            a.x += w * x.x;
            a.y += w * x.y;
            a.z += w * x.z;
            a.w += w * x.w;
        }
        __half2 *dst = reinterpret_cast<__half2 *>(ob + (int64_t)row * D + 4 * d4);
        dst[0] = __floats2half2_rn(a.x, a.y);
        dst[1] = __floats2half2_rn(a.z, a.w);
    }
}

constexpr int kMaxDevices = 64;

template <int D>
int blocks_per_sm(const LaunchCtx &ctx) {
    using C = PrefillCfg<D>;
    static int occ[kMaxDevices] = {0};
    if (ctx.device < 0 || ctx.device >= kMaxDevices) return -1;
    if (occ[ctx.device] == 0) {
        if (cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
            cudaSuccess)
            return -1;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefill_kernel<D>, C::THREADS, C::SMEM) !=
                cudaSuccess ||
            n < 1)
            return -1;
        occ[ctx.device] = n;
    }
    return occ[ctx.device];
}

// Context splits per item: enough CTAs to cover the GPU's resident slots,
// at least two tiles per split, at most kPrefillMaxSplits (or the forced value).
template <int D>
int splits_for(const gqaq_dims &dm, int q_len, const LaunchCtx &ctx) {
    const int occ = blocks_per_sm<D>(ctx);
    if (occ < 1) return -1;
    const int64_t items = prefill_items(dm, q_len);
    if (ctx.prefill_splits > 0) return ctx.prefill_splits < kPrefillMaxSplits ? ctx.prefill_splits : kPrefillMaxSplits;
    const int64_t slots = (int64_t)occ * ctx.num_sms;
    int64_t s = (slots + items - 1) / items;
    const int64_t tiles = ((int64_t)dm.max_len + PrefillCfg<D>::TT - 1) / PrefillCfg<D>::TT;
    const int64_t cap = tiles / 2 > 1 ? tiles / 2 : 1;
    if (s > cap) s = cap;
    if (s > kPrefillMaxSplits) s = kPrefillMaxSplits;
    return (int)(s < 1 ? 1 : s);
}

template <int D>
size_t ws_bytes(const gqaq_dims &dm, int q_len, const LaunchCtx &ctx) {
    const int s = splits_for<D>(dm, q_len, ctx);
    if (s < 1) return 0;
    const int64_t items = prefill_items(dm, q_len);
    const size_t zero = ((size_t)items * 4 + 255) / 256 * 256;
    return zero + (s > 1 ? (size_t)items * s * PrefillCfg<D>::RB * (D + 2) * sizeof(float) : 0);
}

template <int D>
int launch_d(const PrefillArgs &a, const LaunchCtx &ctx) {
    using C = PrefillCfg<D>;
    const gqaq_dims &dm = *a.dims;
    const int splits = splits_for<D>(dm, a.q_len, ctx);
    if (splits < 1) return GQAQ_ERR_CUDA;
    const size_t need = ws_bytes<D>(dm, a.q_len, ctx);
    if (a.workspace == nullptr || a.workspace_bytes < need) return GQAQ_ERR_WORKSPACE;
    const int64_t items = prefill_items(dm, a.q_len);
    if (items * splits > INT32_MAX) return GQAQ_ERR_UNSUPPORTED;

    const uint64_t rows = (uint64_t)dm.batch * dm.num_kv_heads * dm.max_len;
    CUtensorMap kmap, vmap;
    if (!encode_tensor_map_2d(&kmap, a.k_cache, rows, D, 64, C::TT, true)) return GQAQ_ERR_CUDA;
    if (!encode_tensor_map_2d(&vmap, a.v_cache, rows, D, 64, C::TT, true)) return GQAQ_ERR_CUDA;

    PrefillParams p;
    p.q = a.q;
    p.out = a.out;
    p.start = a.start;
    const size_t zero = ((size_t)items * 4 + 255) / 256 * 256;
    p.count = reinterpret_cast<unsigned *>(a.workspace);
    p.part = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(a.workspace) + zero);
    p.status = ctx.status;
    p.B = dm.batch;
    p.Hkv = dm.num_kv_heads;
    p.Lmax = dm.max_len;
    p.q_len = a.q_len;
    p.R = (dm.num_q_heads / dm.num_kv_heads) * a.q_len;
    p.nrb = (p.R + C::RB - 1) / C::RB;
    p.splits = splits;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.timeout_ns = ctx.timeout_ns;
    p.test_stall = ctx.test_stall;
    if (launch_kernel(prefill_kernel<D>, dim3((unsigned)(items * splits)), dim3(C::THREADS), C::SMEM, ctx, 0, kmap,
                      vmap, p) != cudaSuccess)
        return GQAQ_ERR_CUDA;
    return GQAQ_OK;
}

}  // namespace

int64_t prefill_items(const gqaq_dims &dm, int q_len) {
    const int64_t R = (int64_t)(dm.num_q_heads / dm.num_kv_heads) * q_len;
    return (int64_t)dm.batch * dm.num_kv_heads * ((R + 127) / 128);
}

int launch_prefill(const PrefillArgs &a, const LaunchCtx &ctx) {
    switch (a.dims->head_dim) {
        case 64: return launch_d<64>(a, ctx);
        case 128: return launch_d<128>(a, ctx);
        default: return GQAQ_ERR_UNSUPPORTED;
    }
}

size_t prefill_workspace_bytes(const gqaq_dims *dims, int q_len, const LaunchCtx &ctx) {
    switch (dims->head_dim) {
        case 64: return ws_bytes<64>(*dims, q_len, ctx);
        case 128: return ws_bytes<128>(*dims, q_len, ctx);
        default: return 0;
    }
}

}  // namespace gqaq
