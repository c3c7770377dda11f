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

// ===========================================================================
// Tensor-memory kernel (tcgen05): the same work items, splits and merge as
// prefill_kernel, with both products on the 5th-generation tensor cores.
//  - warp 8 (TMA): the item's Q block once, then K and V tiles of 128 tokens
//    (128-byte-swizzled 64-column boxes) into a 3-5 stage ring.
//  - warp 9 (MMA, one thread): S_j = Q K_j^T (M = 128 rows, N = 128 tokens,
//    K = D; both operands K-major in shared memory) into one of three TMEM S
//    buffers, and O += P_j V_j (A = P_j from TMEM, B = V_j MN-major in shared
//    memory, N = D across the 64-channel blocks) into the TMEM O block. Each
//    product is issued as soon as its inputs are there (S_j when tile j has
//    landed, PV_j when its P is written), except that S_j waits for the issue
//    of PV_{j-3}, which reads the P held in the same S buffer (the tensor core
//    runs one thread's MMAs in order). Descriptors are computed once; a stage
//    or K-step is an offset. Completions arrive on mbarriers through
//    tcgen05.commit.
//  - warps 0-7 (softmax): all eight on every tile, warp w on the rows of its
//    TMEM lane quarter (w % 4) and the 64-token half w / 4 of the tile: read
//    the scores from TMEM, mask the causal limit, take P = 2^(x - m_ref)
//    against the row's reference max without a max pass (a half whose P sum
//    stays <= 2^12 needs nothing more; otherwise, for every thread at once,
//    the row's max over both halves becomes the reference and O in TMEM is
//    rescaled), and write P as fp16 inside the columns the half read. Two
//    softmax warps per sub-partition work on the same tile while the tensor
//    core computes the next tile's S into the other buffer.
//  - TMEM (512 columns): O at column 0 (D columns), S buffer b (of three) at
//    128 + 128 b: S_j goes to buffer j % 3 once PV_{j-3} has been issued.
// ===========================================================================
template <int D>
struct TcCfg {
    static constexpr int THREADS = 320;           // 2 softmax warpgroups, TMA warp, MMA warp
    static constexpr int RB = 128;                // rows per item (TMEM lanes)
    static constexpr int TT = 128;                // tokens per stage (N of S)
    static constexpr int KH = D / 64;
    static constexpr int KBLK = TT * 128;         // one 64-column block of a K or V tile
    static constexpr int KBYTES = KH * KBLK;      // = TT * D * 2
    static constexpr int STAGE = 2 * KBYTES;
    static constexpr int QBLK = RB * 128;
    static constexpr int QBYTES = KH * QBLK;
    static constexpr int NSTAGE = D == 128 ? 3 : 5;
    static constexpr int MISC = 2048;             // barriers, flags, and group 1's (m, l) per row at +512
    static constexpr int SMEM = 1024 + QBYTES + NSTAGE * STAGE + MISC;
    static constexpr int TMEM_COLS = 512;
    static constexpr int O_COL = 0, S_COL = 128;  // O (D columns), then S buffer b at 128 + 128 b
    static constexpr int NSB = 3;                 // S buffers: three tiles between S and PV
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(RB * kPrefillMaxSplits * 4 <= NSTAGE * STAGE, "merge weights fit the idle ring");
};

// Shared-memory matrix descriptor: 128-byte swizzle, SBO = 1024 (8 rows of
// 128 B), LBO = lbo (the MN-direction block stride of an MN-major operand;
// not used by K-major operands whose K slice stays inside one 128-byte row).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 D, M x N, B K- or MN-major.
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N, int b_mn_major) {
    return (1u << 4) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, int acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                 "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, int acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
                 "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 64 consecutive columns of this thread's lane: two x32 loads, one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr + 32u));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Barrier 2 over the 256 softmax threads that also reduces a predicate:
// true on every thread when any of them passed true.
__device__ __forceinline__ bool bar_any_256(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, 2, 256, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

// One warp's bounded wait (lane 0 waits, the warp follows): false on timeout or abort.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const PrefillParams &p,
                                          volatile int *abort_flag, int lane) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait(bar, parity, p.timeout_ns, abort_flag);
    return __shfl_sync(0xffffffffu, ok, 0);
}

template <int D>
__global__ void __launch_bounds__(TcCfg<D>::THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
    using C = TcCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sq = smem;
    uint8_t *stages = sq + C::QBYTES;
    // Each stage holds a K tile and a V tile with barriers of their own: a K
    // half is reloaded once its S has completed, a V half once its PV has.
    uint64_t *full = reinterpret_cast<uint64_t *>(stages + C::NSTAGE * C::STAGE);  // K landed
    uint64_t *empty = full + C::NSTAGE;                                           // K free (S done)
    uint64_t *vfull = empty + C::NSTAGE;                                          // V landed
    uint64_t *vempty = vfull + C::NSTAGE;                                         // V free (PV done)
    uint64_t *qbar = vempty + C::NSTAGE;
    uint64_t *s_ready = qbar + 1;          // [NSB]: S_j complete, on s_ready[j % NSB]
    uint64_t *p_ready = s_ready + C::NSB;  // [NSB]: P_j written, on p_ready[j % NSB]
    uint64_t *o_done = p_ready + C::NSB;   // [2]: PV_j completes on o_done[j & 1]
    uint64_t *drain = o_done + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
    int *last_flag = reinterpret_cast<int *>(tslot + 2);
    float *wbuf = reinterpret_cast<float *>(stages);  // merge weights, once the ring is idle

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 8 && lane == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
            mbar_init(smem_u32(&vfull[s]), 1);
            mbar_init(smem_u32(&vempty[s]), 1);
        }
        mbar_init(smem_u32(qbar), 1);
        for (int b = 0; b < C::NSB; ++b) {
            mbar_init(smem_u32(&s_ready[b]), 1);
            mbar_init(smem_u32(&p_ready[b]), 8);  // one arrival per softmax warp
        }
        mbar_init(smem_u32(&o_done[0]), 1);
        mbar_init(smem_u32(&o_done[1]), 1);
        mbar_init(smem_u32(drain), 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    if (warp == 9) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "n"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    pdl_wait_and_release();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

    // ---- the work item and this CTA's slice of its context tiles ----
    const int item = blockIdx.x / p.splits, split = blockIdx.x - (blockIdx.x / p.splits) * p.splits;
    const int rb = item % p.nrb, unit = item / p.nrb;  // unit = b * Hkv + kv
    const int b = unit / p.Hkv;
    const int rho0 = rb * C::RB;
    const int nrows = (p.R - rho0) < C::RB ? (p.R - rho0) : C::RB;
    const int st = p.start[b];
    const bool good = st >= 0 && st <= p.Lmax - p.q_len;
    if (!good && threadIdx.x == 0 && split == 0 && rb == 0 && unit % p.Hkv == 0) raise_flag(p.status, GQAQ_DEV_BAD_POS);
    const int t_first = rho0 % p.q_len, t_last = (rho0 + nrows - 1) % p.q_len;
    const bool wraps = nrows >= p.q_len || t_first > t_last;
    const int t_max = wraps ? p.q_len - 1 : t_last, t_min = wraps ? 0 : t_first;
    const int nt = good ? (st + t_max + C::TT) / C::TT : 0;
    const int j0 = (int)(((int64_t)split * nt) / p.splits), j1 = (int)(((int64_t)(split + 1) * nt) / p.splits);
    const int n = j1 - j0;
    const int kv_end = st + p.q_len;

    if (warp == 8) {
        // ------------------------------------------------------------------
        // TMA producer
        // ------------------------------------------------------------------
        if (lane == 0 && n > 0 && !p.test_stall) {
            const uint64_t pol = l2_policy_evict_first();
            mbar_arrive_expect_tx(smem_u32(qbar), (uint32_t)C::QBYTES);
            const int qrow = unit * p.R + rho0;
#pragma unroll
            for (int kh = 0; kh < C::KH; ++kh)
                tma_load_2d(smem_u32(sq) + kh * C::QBLK, &qmap, 64 * kh, qrow, smem_u32(qbar), pol);
            // K tile ik and V tile iv, each as soon as its half of the stage is
            // free; K leads (S needs it first), V follows.
            int ik = 0, iv = 0;
            bool failed = false;
            uint64_t t_last = global_timer_ns();
            while (iv < n && !failed) {
                bool progressed = false;
                if (ik < n) {
                    const int s = ik % C::NSTAGE;
                    if (ik < C::NSTAGE || mbar_try_wait_ns(smem_u32(&empty[s]), ((uint32_t)(ik / C::NSTAGE) & 1u) ^ 1u,
                                                           iv < ik ? 100u : 2000u)) {
                        const uint32_t kdst = smem_u32(stages + s * C::STAGE), fb = smem_u32(&full[s]);
                        mbar_arrive_expect_tx(fb, (uint32_t)C::KBYTES);
                        const int y = unit * p.Lmax + (j0 + ik) * C::TT;
#pragma unroll
                        for (int kh = 0; kh < C::KH; ++kh) tma_load_2d(kdst + kh * C::KBLK, &kmap, 64 * kh, y, fb, pol);
                        ++ik;
                        progressed = true;
                    }
                }
                if (iv < ik) {
                    const int s = iv % C::NSTAGE;
                    if (iv < C::NSTAGE || mbar_try_wait_ns(smem_u32(&vempty[s]), ((uint32_t)(iv / C::NSTAGE) & 1u) ^ 1u,
                                                           ik < n ? 100u : 2000u)) {
                        const uint32_t vdst = smem_u32(stages + s * C::STAGE) + C::KBYTES, fb = smem_u32(&vfull[s]);
                        mbar_arrive_expect_tx(fb, (uint32_t)C::KBYTES);
                        const int y = unit * p.Lmax + (j0 + iv) * C::TT;
#pragma unroll
                        for (int kh = 0; kh < C::KH; ++kh) tma_load_2d(vdst + kh * C::KBLK, &vmap, 64 * kh, y, fb, pol);
                        ++iv;
                        progressed = true;
                    }
                }
                const uint64_t now = global_timer_ns();
                if (progressed) {
                    t_last = now;
                } else if (*abort_flag || now - t_last >= p.timeout_ns) {
                    failed = true;
                }
            }
            if (failed) {
                raise_flag(p.status, GQAQ_DEV_TIMEOUT);
                *abort_flag = 1;
                // let every copy already issued land before this CTA may retire
                for (int it = ik - C::NSTAGE > 0 ? ik - C::NSTAGE : 0; it < ik; ++it)
                    mbar_wait(smem_u32(&full[it % C::NSTAGE]), (uint32_t)(it / C::NSTAGE) & 1u, p.timeout_ns, nullptr);
                for (int it = iv - C::NSTAGE > 0 ? iv - C::NSTAGE : 0; it < iv; ++it)
                    mbar_wait(smem_u32(&vfull[it % C::NSTAGE]), (uint32_t)(it / C::NSTAGE) & 1u, p.timeout_ns, nullptr);
                mbar_wait(smem_u32(qbar), 0u, p.timeout_ns, nullptr);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------------
        // MMA issuer (one thread)
        // ------------------------------------------------------------------
        if (lane == 0) {
            bool fail = false;
            if (n > 0) {
                fail = !mbar_wait(smem_u32(qbar), 0u, p.timeout_ns, abort_flag);
                constexpr uint32_t IDESC_S = umma_idesc(128, C::TT, 0);
                constexpr uint32_t IDESC_O = umma_idesc(128, D, 1);
                // Descriptors of the Q block and of stage 0's K and V tiles; a stage,
                // a K-step or a block is an offset added to the address field.
                const uint64_t qdesc0 = umma_desc(smem_u32(sq), 16);
                const uint64_t kdesc0 = umma_desc(smem_u32(stages), 16);
                const uint64_t vdesc0 = umma_desc(smem_u32(stages) + C::KBYTES, C::KBLK);
                // Issue each product as soon as its inputs are there: S_is when
                // its K/V tile has landed (and PV_{is-2}, which reads the P held
                // in the same S buffer, is issued: the tensor core runs one
                // thread's MMAs in order), PV_ip when its softmax has written P.
                // A PV never waits for the next tile's load.
                int is = 0, ip = 0;
                uint64_t t_last = global_timer_ns();
                while (ip < n && !fail) {
                    bool progressed = false;
                    const bool s_ok = is < n && ip >= is - (C::NSB - 1);  // PV_{is-NSB} issued: its buffer is free
                    if (s_ok) {
                        const int s = is % C::NSTAGE;
                        if (mbar_try_wait_ns(smem_u32(&full[s]), (uint32_t)(is / C::NSTAGE) & 1u, ip < is ? 100u : 2000u)) {
                            tc_fence_after();
                            // K-step ks: 16 columns of Q and K, 32 B further along the 128-byte
                            // row, a 64-column block further every 4 steps (the descriptor's
                            // address field counts 16-byte units; no carry leaves it).
                            const uint64_t kd = kdesc0 + (uint64_t)((s * C::STAGE) >> 4);
                            const uint32_t sd = tbase + C::S_COL + 128u * (uint32_t)(is % C::NSB);
#pragma unroll
                            for (int ks = 0; ks < D / 16; ++ks)
                                umma_ss(sd, qdesc0 + (uint64_t)(((ks >> 2) * C::QBLK + (ks & 3) * 32) >> 4),
                                        kd + (uint64_t)(((ks >> 2) * C::KBLK + (ks & 3) * 32) >> 4), IDESC_S, ks > 0);
                            umma_commit(smem_u32(&s_ready[is % C::NSB]));
                            umma_commit(smem_u32(&empty[s]));  // the K half is free once S has read it
                            ++is;
                            progressed = true;
                        }
                    }
                    if (ip < is &&
                        mbar_try_wait_ns(smem_u32(&p_ready[ip % C::NSB]), (uint32_t)(ip / C::NSB) & 1u, s_ok ? 100u : 2000u) &&
                        mbar_try_wait_ns(smem_u32(&vfull[ip % C::NSTAGE]), (uint32_t)(ip / C::NSTAGE) & 1u, 100u)) {
                        tc_fence_after();
                        const int s = ip % C::NSTAGE;
                        // K-step kk: 16 tokens (rows 16 kk .. of V, 8 TMEM columns of P);
                        // N = D spans the 64-channel blocks of V through the MN-major
                        // descriptor's leading byte offset (one block = KBLK bytes).
                        const uint64_t vd = vdesc0 + (uint64_t)((s * C::STAGE) >> 4);
                        const uint32_t od = tbase + C::O_COL;
                        const uint32_t pd = tbase + C::S_COL + 128u * (uint32_t)(ip % C::NSB);
                        // P of tokens 0-63 sits in S columns 0-31, of tokens 64-127 in 64-95
                        // (each softmax half writes inside the columns it read)
#pragma unroll
                        for (int kk = 0; kk < C::TT / 16; ++kk)
                            umma_ts(od, pd + 8u * kk + (kk >= 4 ? 32u : 0u), vd + (uint64_t)((kk * 16 * 128) >> 4),
                                    IDESC_O, (ip > 0 || kk > 0) ? 1 : 0);  // the first PV starts O
                        umma_commit(smem_u32(&o_done[ip & 1]));
                        umma_commit(smem_u32(&vempty[s]));
                        ++ip;
                        progressed = true;
                    }
                    const uint64_t now = global_timer_ns();
                    if (progressed) {
                        t_last = now;
                    } else if (*abort_flag || now - t_last >= p.timeout_ns) {
                        fail = true;
                    }
                }
            }
            if (fail) {
                raise_flag(p.status, GQAQ_DEV_TIMEOUT);
                *abort_flag = 1;
            }
            // every issued MMA completes before TMEM is released
            if (n > 0) {
                umma_commit(smem_u32(drain));
                mbar_wait(smem_u32(drain), 0u, p.timeout_ns, nullptr);
            }
        }
    } else {
        // ------------------------------------------------------------------
        // Softmax, all eight warps on every tile: warp w takes the row block
        // of its TMEM lane quarter (w % 4) and column half h = w / 4 of the
        // tile (64 tokens), so the two warps of a sub-partition work on the
        // same tile. Both halves of a row share its reference max m_ref and
        // keep partial sums l; they agree through shared memory, and only when
        // some chunk leaves the fast path (a predicate-reducing barrier per
        // tile tells every thread). P of half h goes to S columns 64 h .. +31,
        // inside the columns it read. One O for the item: a rescale first
        // waits for the previous PV (the only one that can still write O).
        // ------------------------------------------------------------------
        const int half = warp >> 2;
        const int tid = threadIdx.x & 127;
        const bool live = tid < nrows;
        const int lim = st + (rho0 + tid) % p.q_len;
        const uint32_t trow = tbase + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t ocol = trow + C::O_COL + (uint32_t)(half * (D / 2));  // this half's O columns
        float *xchg = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(full) + 512);  // [2][128] misc region
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        // PV_j's completion, on o_done[j & 1]. A parity wait is exact only
        // while the barrier is at most one phase behind: PV_{j-2} complete and
        // PV_{j+2} not issued. The slow path asks for PV_{idx-1} once S_idx is
        // complete, which (in-order MMAs, S_idx issued after PV_{idx-3})
        // implies PV_{idx-3} complete; PV_{idx+1} needs this thread's P. The
        // epilogue asks for PV_{n-2} first (S_{n-1} complete implies PV_{n-4})
        // and then PV_{n-1}.
        auto wait_pv = [&](int j) {
            return warp_wait(smem_u32(&o_done[j & 1]), (uint32_t)(j >> 1) & 1u, p, abort_flag, lane);
        };
        auto fail = [&]() {
            if (lane == 0) {
                raise_flag(p.status, GQAQ_DEV_TIMEOUT);
                *abort_flag = 1;
            }
        };
        for (int idx = 0; idx < n; ++idx) {
            // every thread of the 256 reaches the same barriers each tile, also after a timeout
            ok = ok && warp_wait(smem_u32(&s_ready[idx % C::NSB]), (uint32_t)(idx / C::NSB) & 1u, p, abort_flag, lane);
            if (!ok) fail();
            tc_fence_after();
            const int tok0 = (j0 + idx) * C::TT + 64 * half;  // this half's first token
            const bool need_mask = tok0 + 63 > st + t_min;  // uniform over the item
            const uint32_t sbuf = trow + C::S_COL + 128u * (uint32_t)(idx % C::NSB);
            const uint32_t scol = sbuf + 64u * half;
            uint32_t v[64], pk[32];
            if (ok) {
                tmem_ld64(scol, v);
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) v[e] = 0u;
            }
            // With a positive scale it folds into the exponent's FFMA (mul);
            // otherwise the scores are scaled first (mul = 1).
            float mul = p.scale_log2;
            if (p.scale_log2 <= 0.f) {
#pragma unroll
                for (int e = 0; e < 64; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * p.scale_log2);
                mul = 1.f;
            }
            if (need_mask) {
#pragma unroll
                for (int e = 0; e < 64; ++e)
                    if (tok0 + e > lim) v[e] = __float_as_uint(-INFINITY);
            }
            // P of this half against reference `ref` into pk; returns its sum
            auto half_p = [&](float ref) {
                const float nref = ref == -INFINITY ? 0.f : -ref;
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float e0 = fast_exp2(fmaf(__uint_as_float(v[e]), mul, nref));
                    const float e1 = fast_exp2(fmaf(__uint_as_float(v[e + 1]), mul, nref));
                    s4[(e >> 1) & 3] += e0 + e1;
                    pk[e >> 1] = pack_half2(e0, e1);
                }
                return (s4[0] + s4[1]) + (s4[2] + s4[3]);
            };
            // Fast path: P against the current reference; the half's sum bounds
            // every P in it, so a sum <= 2^12 means every P fits fp16.
            float cs = 0.f;
            if (m_ref != -INFINITY) cs = half_p(m_ref);
            const bool redo = m_ref == -INFINITY || cs > 4096.f;
            if (bar_any_256(redo)) {
                // Slow path (the first tiles, or a score well above the reference):
                // the row's max over both halves becomes the reference; l, O and
                // this half's P follow it.
                float r4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < 64; ++e) r4[e & 3] = fmaxf(r4[e & 3], __uint_as_float(v[e]));
                xchg[half * 128 + tid] = fmaxf(fmaxf(r4[0], r4[1]), fmaxf(r4[2], r4[3])) * mul;
                named_bar_sync(2, 256);
                const float cm = fmaxf(xchg[tid], xchg[128 + tid]);
                const bool up = cm > m_ref;
                const float alpha = up ? fast_exp2(m_ref - cm) : 1.f;  // 0 when m_ref is -inf
                if (up) {
                    m_ref = cm;
                    l *= alpha;
                }
                if (__any_sync(0xffffffffu, up && idx >= 1)) {  // O holds earlier tiles
                    ok = ok && wait_pv(idx - 1);                  // the last PV that writes O
                    if (!ok) fail();
                    tc_fence_after();
                    if (ok) {
#pragma unroll 1
                        for (int oc = 0; oc < D / 64; ++oc) {
                            uint32_t o[32];
                            tmem_ld32(ocol + 32u * oc, o);
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(ocol + 32u * oc, o);
                        }
                        tmem_wait_st();
                    }
                }
                cs = half_p(m_ref);
            }
            l += cs;
            if (ok) {
                tmem_st32(scol, pk);  // P over this half's columns (the first 32 of the 64 it read)
                tmem_wait_st();
            }
            if (ok && (j0 + idx) * C::TT + C::TT > kv_end) {  // uniform: wait for this tile's V to land
                ok = warp_wait(smem_u32(&vfull[idx % C::NSTAGE]), (uint32_t)(idx / C::NSTAGE) & 1u, p, abort_flag, lane);
                if (!ok) fail();
            }
            const int vrow_tok = (j0 + idx) * C::TT + tid;
            if (ok && (j0 + idx) * C::TT + C::TT > kv_end && vrow_tok >= kv_end && half < C::KH) {
                // rows past the chunk may hold anything: zero them so 0 * NaN cannot
                // reach O (half h clears the row's 64-channel block h)
                uint8_t *vrow = stages + (idx % C::NSTAGE) * C::STAGE + C::KBYTES + half * C::KBLK + tid * 128;
#pragma unroll
                for (int q16 = 0; q16 < 8; ++q16)
                    *reinterpret_cast<uint4 *>(vrow + 16 * q16) = make_uint4(0u, 0u, 0u, 0u);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // zeroed rows reach the tensor core
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&p_ready[idx % C::NSB]));
        }
        // ---- epilogue: O after the last PV; l of both halves; each half writes its columns ----
        if (ok && n > 1) {
            ok = wait_pv(n - 2);
            if (!ok) fail();
        }
        if (ok && n > 0) {
            ok = wait_pv(n - 1);  // every PV is done (in-order completion)
            if (!ok) fail();
        }
        tc_fence_after();
        xchg[half * 128 + tid] = l;
        named_bar_sync(2, 256);
        const float L = xchg[tid] + xchg[128 + tid];
        const float inv = L > 0.f ? 1.f / L : 0.f;
        __half *ob = p.out + ((int64_t)unit * p.R + rho0) * D;
        float *pml = p.part + (int64_t)blockIdx.x * C::RB * (D + 2);
        float *pacc = pml + 2 * C::RB;
        if (p.splits > 1 && live && half == 0) reinterpret_cast<float2 *>(pml)[tid] = make_float2(m_ref, L);
#pragma unroll 1
        for (int ch = 0; ch < D / 64; ++ch) {
            const int c0 = half * (D / 2) + 32 * ch;  // output channel of column e: c0 + e
            uint32_t v[32];
            if (ok && n > 0) {
                tmem_ld32(trow + C::O_COL + (uint32_t)c0, v);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
            if (!live) continue;
            if (p.splits == 1) {
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint4 h;
                    h.x = pack_half2(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv);
                    h.y = pack_half2(__uint_as_float(v[e + 2]) * inv, __uint_as_float(v[e + 3]) * inv);
                    h.z = pack_half2(__uint_as_float(v[e + 4]) * inv, __uint_as_float(v[e + 5]) * inv);
                    h.w = pack_half2(__uint_as_float(v[e + 6]) * inv, __uint_as_float(v[e + 7]) * inv);
                    *reinterpret_cast<uint4 *>(ob + (int64_t)tid * D + c0 + e) = h;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(pacc + (int64_t)tid * D + c0 + e) =
                        make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                    __uint_as_float(v[e + 3]));
            }
        }
    }

    // ---- all roles meet: the ring is idle, every MMA has completed ----
    tc_fence_before();
    __syncthreads();
    if (warp == 9) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "n"(C::TMEM_COLS));
    if (p.splits == 1 || warp >= 4) return;

    // ---- split: arrival, and the last arrival's merge (softmax group 0, 128 threads) ----
    constexpr int NCT = 128;
    const int tid = threadIdx.x;
    if (tid == 0) {
        // __syncthreads above orders every thread's partial stores before this
        // release; the item's last arrival acquires all of them.
        const unsigned old = atomic_add_acq_rel_gpu(&p.count[item], 1u);
        const int last = old + 1u == (unsigned)p.splits;
        if (last) p.count[item] = 0u;
        *last_flag = last;
    }
    named_bar_sync(1, NCT);
    if (!*last_flag) return;
    __half *ob = p.out + ((int64_t)unit * p.R + rho0) * D;
    const float *base = p.part + (int64_t)item * p.splits * C::RB * (D + 2);
    for (int row = tid; row < nrows; row += NCT) {
        float mst = -INFINITY;
        for (int sp = 0; sp < p.splits; ++sp)
            mst = fmaxf(mst, __ldcg(base + (int64_t)sp * C::RB * (D + 2) + 2 * row));
        float L = 0.f;
        for (int sp = 0; sp < p.splits; ++sp) {
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(base + (int64_t)sp * C::RB * (D + 2)) + row);
            const float f = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - mst);
            wbuf[row * kPrefillMaxSplits + sp] = f;
            L += f * ml.y;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int sp = 0; sp < p.splits; ++sp) wbuf[row * kPrefillMaxSplits + sp] *= inv;
    }
    named_bar_sync(1, NCT);
    for (int e = tid; e < nrows * (D / 4); e += NCT) {
        const int row = e / (D / 4), d4 = e - (e / (D / 4)) * (D / 4);
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < p.splits; ++sp) {
            const float w = wbuf[row * kPrefillMaxSplits + sp];
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

template <int D, bool TC>
int blocks_per_sm(const LaunchCtx &ctx) {
    static int occ[kMaxDevices] = {0};
    if (ctx.device < 0 || ctx.device >= kMaxDevices) return -1;
    if (occ[ctx.device] == 0) {
        int n = 0;
        cudaError_t e;
        if constexpr (TC) {
            e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<D>::SMEM);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefill_tc_kernel<D>, TcCfg<D>::THREADS,
                                                                  TcCfg<D>::SMEM);
        } else {
            e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, PrefillCfg<D>::SMEM);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefill_kernel<D>, PrefillCfg<D>::THREADS,
                                                                  PrefillCfg<D>::SMEM);
        }
        if (e != cudaSuccess || n < 1) return -1;
        occ[ctx.device] = n;
    }
    return occ[ctx.device];
}

// Context splits per item (or the forced value): the count s <= min(tiles / 2,
// kPrefillMaxSplits) that minimises waves x (tiles per split + 2), i.e.
// ceil(items s / slots) (ceil(tiles / s) + 2), for a context of max_len
// tokens; the 2 stands for a CTA's fixed cost (prologue, epilogue, merge) in
// tile times. Ties go to fewer splits (fewer partials to merge).
template <int D, bool TC>
int splits_for(const gqaq_dims &dm, int q_len, const LaunchCtx &ctx) {
    const int occ = blocks_per_sm<D, TC>(ctx);
    if (occ < 1) return -1;
    const int64_t items = prefill_items(dm, q_len);
    if (ctx.prefill_splits > 0) return ctx.prefill_splits < kPrefillMaxSplits ? ctx.prefill_splits : kPrefillMaxSplits;
    const int64_t slots = (int64_t)occ * ctx.num_sms;
    const int tt = TC ? TcCfg<D>::TT : PrefillCfg<D>::TT;
    const int64_t tiles = ((int64_t)dm.max_len + tt - 1) / tt;
    int64_t cap = tiles / 2 > 1 ? tiles / 2 : 1;
    if (cap > kPrefillMaxSplits) cap = kPrefillMaxSplits;
    int64_t best = 1, best_cost = -1;
    for (int64_t s = 1; s <= cap; ++s) {
        const int64_t cost = ((items * s + slots - 1) / slots) * ((tiles + s - 1) / s + 2);
        if (best_cost < 0 || cost < best_cost) {
            best = s;
            best_cost = cost;
        }
    }
    return (int)best;
}

// Workspace for either kernel: the counters, then partials for the larger split.
template <int D>
size_t ws_bytes(const gqaq_dims &dm, int q_len, const LaunchCtx &ctx) {
    const int s0 = splits_for<D, false>(dm, q_len, ctx), s1 = splits_for<D, true>(dm, q_len, ctx);
    if (s0 < 1 || s1 < 1) return 0;
    const int s = s0 > s1 ? s0 : s1;
    const int64_t items = prefill_items(dm, q_len);
    const size_t zero = ((size_t)items * 4 + 255) / 256 * 256;
    return zero + (s > 1 ? (size_t)items * s * PrefillCfg<D>::RB * (D + 2) * sizeof(float) : 0);
}

template <int D, bool TC>
int launch_d(const PrefillArgs &a, const LaunchCtx &ctx) {
    using C = PrefillCfg<D>;
    const gqaq_dims &dm = *a.dims;
    const int splits = splits_for<D, TC>(dm, a.q_len, ctx);
    if (splits < 1) return GQAQ_ERR_CUDA;
    const size_t need = ws_bytes<D>(dm, a.q_len, ctx);
    if (a.workspace == nullptr || a.workspace_bytes < need) return GQAQ_ERR_WORKSPACE;
    const int64_t items = prefill_items(dm, a.q_len);
    if (items * splits > INT32_MAX) return GQAQ_ERR_UNSUPPORTED;

    const int tt = TC ? TcCfg<D>::TT : C::TT;
    const uint64_t rows = (uint64_t)dm.batch * dm.num_kv_heads * dm.max_len;
    CUtensorMap kmap, vmap, qmap;
    if (!encode_tensor_map_2d(&kmap, a.k_cache, rows, D, 64, tt, true)) return GQAQ_ERR_CUDA;
    if (!encode_tensor_map_2d(&vmap, a.v_cache, rows, D, 64, tt, true)) return GQAQ_ERR_CUDA;

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
    cudaError_t e;
    if constexpr (TC) {
        const uint64_t qrows = (uint64_t)dm.batch * dm.num_kv_heads * p.R;  // [B][Hq][q_len] rows of D
        if (!encode_tensor_map_2d(&qmap, a.q, qrows, D, 64, TcCfg<D>::RB, true)) return GQAQ_ERR_CUDA;
        e = launch_kernel(prefill_tc_kernel<D>, dim3((unsigned)(items * splits)), dim3(TcCfg<D>::THREADS),
                          TcCfg<D>::SMEM, ctx, 0, qmap, kmap, vmap, p);
    } else {
        e = launch_kernel(prefill_kernel<D>, dim3((unsigned)(items * splits)), dim3(C::THREADS), C::SMEM, ctx, 0, kmap,
                          vmap, p);
    }
    return e == cudaSuccess ? GQAQ_OK : GQAQ_ERR_CUDA;
}

template <int D>
int launch_kind(const PrefillArgs &a, const LaunchCtx &ctx) {
    return ctx.prefill_kernel == 2 ? launch_d<D, false>(a, ctx) : launch_d<D, true>(a, ctx);
}

}  // namespace

int64_t prefill_items(const gqaq_dims &dm, int q_len) {
    const int64_t R = (int64_t)(dm.num_q_heads / dm.num_kv_heads) * q_len;
    return (int64_t)dm.batch * dm.num_kv_heads * ((R + 127) / 128);
}

int launch_prefill(const PrefillArgs &a, const LaunchCtx &ctx) {
    switch (a.dims->head_dim) {
        case 64: return launch_kind<64>(a, ctx);
        case 128: return launch_kind<128>(a, ctx);
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
