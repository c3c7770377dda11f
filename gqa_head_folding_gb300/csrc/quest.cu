// quest.cu -- Quest page metadata, page scores and top-K page selection.
//
// "Quest: Query-Aware Sparsity for Efficient Long-Context LLM Inference"
// (reviewer's summary):
//  - page-score section: per page p and channel i the keys' minimum m_{p,i}
//    and maximum M_{p,i} are kept and updated when a key arrives, and the page
//    score is U(p,q) = sum_i max(q_i m_{p,i}, q_i M_{p,i}), an upper bound of
//    q.k for every key of the page;
//  - token-budget section: K pages are picked per query (budget B = K*S).
// With grouped query heads one page set serves the G query rows of a KV
// head, so a KV head's score is the largest U over its G rows.
//
// The score kernel evaluates U as a plain dot product. Because m <= M,
// max(q_i m_i, q_i M_i) equals min(q_i,0) m_i + max(q_i,0) M_i for every
// sign of q_i. So U = q_neg . m + q_pos . M with q_neg = min(q,0) and
// q_pos = max(q,0), both exact in fp16, against the [m; M] record of 2D
// halves that the metadata stores per page.
#include <math.h>

#include "internal.h"

namespace gqaq {

// ---------------------------------------------------------------------------
// Append one token per (sequence, KV head) and update its page min/max.
// One warp per unit; lane l owns D/32 consecutive channels.
// ---------------------------------------------------------------------------
struct AppendParams {
    __half *k_cache, *v_cache, *meta;
    const __half *k_new, *v_new;
    const int *pos;
    int *status;
    int B, Hkv, Lmax, Pmax, S;
};

template <int D>
__global__ void __launch_bounds__(128) append_kv_kernel(const AppendParams p) {
    pdl_wait_and_release();
    constexpr int EPL = D / 32;
    const int u = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (u >= p.B * p.Hkv) return;
    const int b = u / p.Hkv;
    const int pos = p.pos[b];
    if (pos < 0 || pos >= p.Lmax) {
        if (lane == 0) raise_flag(p.status, GQAQ_DEV_BAD_POS);
        return;
    }
    const int64_t row = (int64_t)u * p.Lmax + pos;
    const int page = pos / p.S;
    __half *mrow = p.meta + ((int64_t)u * p.Pmax + page) * 2 * D;
    const int c0 = lane * EPL;
    __half kn[EPL], vn[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        kn[e] = p.k_new[(int64_t)u * D + c0 + e];
        vn[e] = p.v_new[(int64_t)u * D + c0 + e];
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        p.k_cache[row * D + c0 + e] = kn[e];
        p.v_cache[row * D + c0 + e] = vn[e];
    }
    const bool fresh = (pos % p.S) == 0;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        __half mn = kn[e], mx = kn[e];
        if (!fresh) {
            const __half om = mrow[c0 + e], oM = mrow[D + c0 + e];
            const float kf = __half2float(kn[e]);
            mn = (kf < __half2float(om)) ? kn[e] : om;
            mx = (kf > __half2float(oM)) ? kn[e] : oM;
        }
        mrow[c0 + e] = mn;
        mrow[D + c0 + e] = mx;
    }
}

// ---------------------------------------------------------------------------
// Build page min/max from the cache for pages [p0, p1). One warp per page.
// ---------------------------------------------------------------------------
struct MetaParams {
    const __half *k_cache;
    const int *valid_len;
    __half *meta;
    int *status;
    int B, Hkv, Lmax, Pmax, S, p0, p1;
};

template <int D>
__global__ void __launch_bounds__(256) update_meta_kernel(const MetaParams p) {
    pdl_wait_and_release();
    constexpr int EPL = D / 32;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int npg = p.p1 - p.p0;
    const int64_t u = gw / npg;
    if (u >= (int64_t)p.B * p.Hkv) return;
    const int page = p.p0 + (int)(gw - u * npg);
    const int b = (int)(u / p.Hkv);
    const int raw = p.valid_len[b];
    if (lane == 0 && page == p.p0 && (u % p.Hkv) == 0 && (raw < 1 || raw > p.Lmax))
        raise_flag(p.status, GQAQ_DEV_BAD_LEN);
    const int len = clamp_len(raw, p.Lmax);
    const int t0 = page * p.S;
    if (t0 >= len) return;
    const int t1 = (t0 + p.S < len) ? t0 + p.S : len;
    const __half *kr = p.k_cache + ((int64_t)u * p.Lmax) * D + lane * EPL;
    float mn[EPL], mx[EPL];
    __half hmn[EPL], hmx[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        hmn[e] = hmx[e] = kr[(int64_t)t0 * D + e];
        mn[e] = mx[e] = __half2float(hmn[e]);
    }
    for (int t = t0 + 1; t < t1; ++t) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const __half x = kr[(int64_t)t * D + e];
            const float xf = __half2float(x);
            if (xf < mn[e]) { mn[e] = xf; hmn[e] = x; }
            if (xf > mx[e]) { mx[e] = xf; hmx[e] = x; }
        }
    }
    __half *mrow = p.meta + (u * p.Pmax + page) * 2 * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        mrow[e] = hmn[e];
        mrow[D + e] = hmx[e];
    }
}

// ---------------------------------------------------------------------------
// Page scores. Persistent CTAs over a balanced split of 64-page tiles.
// warp 8 streams metadata tiles with TMA (128-byte swizzle). Consumer warp w
// scores pages 8w..8w+7 of a tile: lane = 8*quarter + page. Each lane
// covers one quarter of the page's [m; M] record against the matching
// quarter of [q_neg; q_pos].
// ---------------------------------------------------------------------------
template <int D, int G>
struct ScoreCfg {
    static constexpr int NCW = 8;
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int TILE = 64;                  // pages per stage
    static constexpr int PPW = 8;                    // pages per consumer warp
    static constexpr int NB = 2 * D / 64;            // 128-byte column blocks per record
    static constexpr int BLK = TILE * 128;
    static constexpr int STAGE = NB * BLK;           // = TILE * 4 * D bytes
    static constexpr int NSTAGE = 4;
    static constexpr int QT_BYTES = G * 2 * D * 2;   // [G][2D] fp16 q_neg | q_pos
    static constexpr int SMEM = 1024 + NSTAGE * STAGE + QT_BYTES + 256;
    static constexpr int NCHQ = D / 16;              // 16-byte chunks per quarter
    static constexpr bool QREG = (G * D <= 512);
    static constexpr int GQ = QREG ? G : 4;
    static constexpr int NPASS = G / GQ;
};

struct ScoreParams {
    const __half *q;
    const int *valid_len;
    float *scores;
    int *status;
    int B, Hkv, Lmax, Pmax, S;
    uint64_t timeout_ns;
};

__device__ __forceinline__ uint32_t hmin0(uint32_t x) {
    __half2 h = *reinterpret_cast<__half2 *>(&x);
    __half2 r = __hmin2(h, __float2half2_rn(0.f));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t hmax0(uint32_t x) {
    __half2 h = *reinterpret_cast<__half2 *>(&x);
    __half2 r = __hmax2(h, __float2half2_rn(0.f));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint4 clamp_chunk(uint4 v, bool neg) {
    return neg ? make_uint4(hmin0(v.x), hmin0(v.y), hmin0(v.z), hmin0(v.w))
               : make_uint4(hmax0(v.x), hmax0(v.y), hmax0(v.z), hmax0(v.w));
}

template <int D, int G>
__global__ void __launch_bounds__(ScoreCfg<D, G>::THREADS, 1)
    score_pages_kernel(const __grid_constant__ CUtensorMap mmap, const ScoreParams p) {
    using C = ScoreCfg<D, G>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __half *qt_s = reinterpret_cast<__half *>(smem + C::NSTAGE * C::STAGE);
    uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(qt_s) + C::QT_BYTES);
    uint64_t *empty = full + C::NSTAGE;
    int64_t *sch = reinterpret_cast<int64_t *>(empty + C::NSTAGE);  // t_begin, t_end, off_b, b
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sch + 4);

    pdl_wait_and_release();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hq = p.Hkv * G;
    TileRule rule;
    rule.sparse = 0;
    rule.lmax = p.Lmax;
    rule.page_size = p.S;
    rule.kpages = 1;
    rule.tile_tokens = C::TILE * p.S;  // ceil(ceil(L/S)/TILE) == ceil(L/(S*TILE))
    rule.pages_per_tile = 1;

    if (warp == C::NCW) {
        int64_t T, off_b;
        int b;
        locate_tile(p.valid_len, p.B, p.Hkv, rule, 0, T, b, off_b);
        const int64_t tb = tile_begin(blockIdx.x, T, gridDim.x);
        const int64_t te = tile_begin(blockIdx.x + 1, T, gridDim.x);
        if (tb < te) locate_tile(p.valid_len, p.B, p.Hkv, rule, tb, T, b, off_b);
        if (lane == 0) {
            sch[0] = tb;
            sch[1] = te;
            sch[2] = off_b;
            sch[3] = b;
            *abort_flag = 0;
            for (int s = 0; s < C::NSTAGE; ++s) {
                mbar_init(smem_u32(&full[s]), 1);
                mbar_init(smem_u32(&empty[s]), C::NCW);
            }
            fence_mbar_init();
            prefetch_tensormap(&mmap);
        }
    }
    __syncthreads();
    const int64_t t_begin = sch[0], t_end = sch[1];
    if (t_begin >= t_end) return;

    // position of the first tile
    int b = (int)sch[3];
    int tiles_b = rule.tiles(p.valid_len[b]);
    int kv = (int)((t_begin - sch[2]) / tiles_b);
    int local = (int)((t_begin - sch[2]) % tiles_b);

    if (warp == C::NCW) {
        const uint64_t pol = l2_policy_evict_first();
        int i = 0;
        bool failed = false;
        for (int64_t t = t_begin; t < t_end; ++t, ++i) {
            const int s = i % C::NSTAGE;
            const uint32_t ph = (uint32_t)(i / C::NSTAGE) & 1u;
            if (i >= C::NSTAGE) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait(smem_u32(&empty[s]), ph ^ 1u, p.timeout_ns, abort_flag);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { failed = true; break; }
            }
            if (lane == 0) {
                const uint32_t fb = smem_u32(&full[s]);
                const uint32_t dst = smem_u32(smem + s * C::STAGE);
                mbar_arrive_expect_tx(fb, (uint32_t)C::STAGE);
                const int y = (b * p.Hkv + kv) * p.Pmax + local * C::TILE;
#pragma unroll
                for (int kb = 0; kb < C::NB; ++kb) tma_load_2d(dst + kb * C::BLK, &mmap, 64 * kb, y, fb, pol);
            }
            if (++local == tiles_b) {
                local = 0;
                if (++kv == p.Hkv) {
                    kv = 0;
                    do { ++b; tiles_b = (b < p.B) ? rule.tiles(p.valid_len[b]) : 1; } while (b < p.B && tiles_b == 0);
                }
            }
        }
        if (failed && lane == 0) {
            raise_flag(p.status, GQAQ_DEV_TIMEOUT);
            *abort_flag = 1;
            const int first = i - C::NSTAGE > 0 ? i - C::NSTAGE : 0;
            for (int it = first; it < i; ++it)
                mbar_wait(smem_u32(&full[it % C::NSTAGE]), (uint32_t)(it / C::NSTAGE) & 1u, p.timeout_ns, nullptr);
        }
        __syncwarp();
        return;
    }

    // consumers
    const int cw = warp;
    const int jp = lane & 7;          // page within this warp's 8
    const int qq = lane >> 3;         // record quarter: 0,1 = m halves, 2,3 = M halves
    const int row = cw * C::PPW + jp; // page row within the stage
    const int cq0 = qq * (D / 2);     // first record channel of this quarter
    const uint32_t roff = (uint32_t)((cq0 / 64) * C::BLK + row * 128);
    const uint32_t x0 = (uint32_t)(((cq0 % 64) / 8) ^ (row & 7));
    const bool negq = qq < 2;
    const int qch0 = (qq & 1) * (D / 2);  // channel of q matching this quarter

    uint4 qr[C::GQ][C::NCHQ];
    int cur_unit = -1;
    int i = 0;
    for (int64_t t = t_begin; t < t_end; ++t, ++i) {
        const int unit = b * p.Hkv + kv;
        const int len = clamp_len(p.valid_len[b], p.Lmax);
        const int P = (len + p.S - 1) / p.S;
        if (unit != cur_unit) {
            cur_unit = unit;
            const __half *qg = p.q + ((int64_t)b * Hq + (int64_t)kv * G) * D;
            if (C::QREG) {
#pragma unroll
                for (int g = 0; g < C::GQ; ++g)
#pragma unroll
                    for (int c = 0; c < C::NCHQ; ++c)
                        qr[g][c] = clamp_chunk(*reinterpret_cast<const uint4 *>(qg + g * D + qch0 + c * 8), negq);
            } else {
                // all consumers are at the same tile here: rebuild [q_neg | q_pos] in smem
                named_bar_sync(1, C::NCW * 32);
                for (int e = threadIdx.x; e < G * D / 8; e += C::NCW * 32) {
                    const int g = e / (D / 8), c = e % (D / 8);
                    const uint4 v = *reinterpret_cast<const uint4 *>(qg + g * D + c * 8);
                    reinterpret_cast<uint4 *>(qt_s + g * 2 * D)[c] = clamp_chunk(v, true);
                    reinterpret_cast<uint4 *>(qt_s + g * 2 * D + D)[c] = clamp_chunk(v, false);
                }
                named_bar_sync(1, C::NCW * 32);
            }
        }
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
        const int page = local * C::TILE + row;
        if (ok && local * C::TILE + cw * C::PPW < P) {
            const uint32_t base = smem_u32(smem + s * C::STAGE) + roff;
            float u[G];
#pragma unroll
            for (int pass = 0; pass < C::NPASS; ++pass) {
                if (!C::QREG) {
#pragma unroll
                    for (int g = 0; g < C::GQ; ++g)
#pragma unroll
                        for (int c = 0; c < C::NCHQ; ++c)
                            qr[g][c] = lds128(smem_u32(qt_s + (pass * C::GQ + g) * 2 * D + cq0 + c * 8));
                }
                float a0[C::GQ], a1[C::GQ];
#pragma unroll
                for (int g = 0; g < C::GQ; ++g) a0[g] = a1[g] = 0.f;
#pragma unroll
                for (int c = 0; c < C::NCHQ; ++c) {
                    const uint4 mc = lds128(base + ((x0 ^ (uint32_t)c) << 4));
#pragma unroll
                    for (int g = 0; g < C::GQ; ++g) {
                        a0[g] = fma_h_lo(qr[g][c].x, mc.x, a0[g]);
                        a1[g] = fma_h_hi(qr[g][c].x, mc.x, a1[g]);
                        a0[g] = fma_h_lo(qr[g][c].y, mc.y, a0[g]);
                        a1[g] = fma_h_hi(qr[g][c].y, mc.y, a1[g]);
                        a0[g] = fma_h_lo(qr[g][c].z, mc.z, a0[g]);
                        a1[g] = fma_h_hi(qr[g][c].z, mc.z, a1[g]);
                        a0[g] = fma_h_lo(qr[g][c].w, mc.w, a0[g]);
                        a1[g] = fma_h_hi(qr[g][c].w, mc.w, a1[g]);
                    }
                }
#pragma unroll
                for (int g = 0; g < C::GQ; ++g) u[pass * C::GQ + g] = a0[g] + a1[g];
            }
            float best = -INFINITY;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float x = u[g];
                x += __shfl_xor_sync(0xffffffffu, x, 8);
                x += __shfl_xor_sync(0xffffffffu, x, 16);
                best = fmaxf(best, x);
            }
            if (qq == 0 && page < P) p.scores[(int64_t)unit * p.Pmax + page] = best;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        if (++local == tiles_b) {
            local = 0;
            if (++kv == p.Hkv) {
                kv = 0;
                do { ++b; tiles_b = (b < p.B) ? rule.tiles(p.valid_len[b]) : 1; } while (b < p.B && tiles_b == 0);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Top-K pages: one CTA per (KV head, sequence). Order-preserving fp32 -> u32
// keys in shared memory; four 8-bit MSB-first radix passes find the K-th
// largest key; pages above it, plus the lowest-indexed pages equal to it,
// are compacted in ascending page order.
// ---------------------------------------------------------------------------
struct TopkParams {
    const float *scores;
    const int *valid_len;
    int *page_idx;
    int *status;
    int B, Hkv, Lmax, Pmax, S, k;
};

constexpr int kTopkThreads = 512;

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t x = __float_as_uint(f);
    if (x == 0x80000000u) x = 0u;  // -0 ranks with +0
    return (x & 0x80000000u) ? ~x : (x | 0x80000000u);
}

__global__ void __launch_bounds__(kTopkThreads) topk_pages_kernel(const TopkParams p) {
    extern __shared__ uint32_t keys[];
    __shared__ int hist[256];
    __shared__ int sh_digit, sh_rem;
    __shared__ int wsum[2][kTopkThreads / 32];
    pdl_wait_and_release();
    const int kv = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t unit = (int64_t)b * p.Hkv + kv;
    const int len = clamp_len(p.valid_len[b], p.Lmax);
    const int P = (len + p.S - 1) / p.S;
    int *out = p.page_idx + unit * p.k;
    if (P <= p.k) {
        for (int j = tid; j < p.k; j += kTopkThreads) out[j] = j < P ? j : -1;
        return;
    }
    const float *sc = p.scores + unit * p.Pmax;
    for (int i = tid; i < P; i += kTopkThreads) keys[i] = order_key(sc[i]);

    uint32_t prefix = 0, mask = 0;
    int remaining = p.k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
        __syncthreads();
        for (int i = tid; i < P; i += kTopkThreads) {
            const uint32_t key = keys[i];
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (warp == 0) {
            int c[8], s = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                c[e] = hist[255 - 8 * lane - e];
                s += c[e];
            }
            int incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int excl = incl - s;
            if (excl < remaining && remaining <= incl) {
                int cum = excl;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (cum + c[e] >= remaining) {
                        sh_digit = 255 - 8 * lane - e;
                        sh_rem = remaining - cum;
                        break;
                    }
                    cum += c[e];
                }
            }
        }
        __syncthreads();
        prefix |= (uint32_t)sh_digit << shift;
        mask |= 255u << shift;
        remaining = sh_rem;
        __syncthreads();
    }
    const uint32_t kth = prefix;
    const int need_eq = remaining;  // keys equal to kth to take, lowest pages first

    // contiguous chunk per thread, counts of (> kth) and (== kth)
    const int chunk = (P + kTopkThreads - 1) / kTopkThreads;
    const int p0 = tid * chunk < P ? tid * chunk : P;
    const int p1 = p0 + chunk < P ? p0 + chunk : P;
    int n_gt = 0, n_eq = 0;
    for (int i = p0; i < p1; ++i) {
        const uint32_t key = keys[i];
        n_gt += key > kth;
        n_eq += key == kth;
    }
    // block exclusive scan of (n_gt, n_eq)
    int ig = n_gt, ie = n_eq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yg = __shfl_up_sync(0xffffffffu, ig, o);
        const int ye = __shfl_up_sync(0xffffffffu, ie, o);
        if (lane >= o) { ig += yg; ie += ye; }
    }
    if (lane == 31) { wsum[0][warp] = ig; wsum[1][warp] = ie; }
    __syncthreads();
    int bg = 0, be = 0;
    for (int w = 0; w < warp; ++w) { bg += wsum[0][w]; be += wsum[1][w]; }
    const int gt_before = bg + ig - n_gt;
    const int eq_before = be + ie - n_eq;
    int pos = gt_before + (eq_before < need_eq ? eq_before : need_eq);
    int eq_rank = eq_before;
    for (int i = p0; i < p1; ++i) {
        const uint32_t key = keys[i];
        const bool take = key > kth || (key == kth && eq_rank < need_eq);
        eq_rank += key == kth;
        if (take) {
            if (pos < p.k) out[pos] = i;
            ++pos;
        }
    }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
namespace {
constexpr int kMaxDevices = 64;

template <int D>
int launch_append_t(const gqaq_dims *d, __half *kc, __half *vc, __half *meta, const __half *kn,
                    const __half *vn, const int *pos, const LaunchCtx &ctx) {
    AppendParams p;
    p.k_cache = kc; p.v_cache = vc; p.meta = meta; p.k_new = kn; p.v_new = vn; p.pos = pos;
    p.status = ctx.status;
    p.B = d->batch; p.Hkv = d->num_kv_heads; p.Lmax = d->max_len; p.S = d->page_size;
    p.Pmax = (d->max_len + d->page_size - 1) / d->page_size;
    const int units = d->batch * d->num_kv_heads;
    return launch_kernel(append_kv_kernel<D>, dim3((units + 3) / 4), dim3(128), 0, ctx, 0, p) == cudaSuccess
               ? GQAQ_OK
               : GQAQ_ERR_CUDA;
}

template <int D>
int launch_meta_t(const gqaq_dims *d, const __half *kc, const int *vl, __half *meta, int p0, int p1,
                  const LaunchCtx &ctx) {
    MetaParams p;
    p.k_cache = kc; p.valid_len = vl; p.meta = meta; p.status = ctx.status;
    p.B = d->batch; p.Hkv = d->num_kv_heads; p.Lmax = d->max_len; p.S = d->page_size;
    p.Pmax = (d->max_len + d->page_size - 1) / d->page_size;
    p.p0 = p0; p.p1 = p1;
    const int64_t warps = (int64_t)d->batch * d->num_kv_heads * (p1 - p0);
    if (warps == 0) return GQAQ_OK;
    const int64_t blocks = (warps + 7) / 8;
    if (blocks > 0x7fffffff) return GQAQ_ERR_UNSUPPORTED;
    return launch_kernel(update_meta_kernel<D>, dim3((unsigned)blocks), dim3(256), 0, ctx, 0, p) == cudaSuccess
               ? GQAQ_OK
               : GQAQ_ERR_CUDA;
}

template <int D, int G>
int launch_score_t(const gqaq_dims *d, const __half *q, const __half *meta, const int *vl, float *scores,
                   const LaunchCtx &ctx) {
    using C = ScoreCfg<D, G>;
    static int occ[kMaxDevices] = {0};
    if (ctx.device < 0 || ctx.device >= kMaxDevices) return GQAQ_ERR_CUDA;
    auto kern = score_pages_kernel<D, G>;
    if (occ[ctx.device] == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return GQAQ_ERR_CUDA;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::THREADS, C::SMEM) != cudaSuccess || n < 1)
            return GQAQ_ERR_CUDA;
        occ[ctx.device] = n;
    }
    int grid = occ[ctx.device] * ctx.num_sms;
    if (ctx.max_ctas > 0 && ctx.max_ctas < grid) grid = ctx.max_ctas;
    const int Pmax = (d->max_len + d->page_size - 1) / d->page_size;
    const uint64_t rows = (uint64_t)d->batch * d->num_kv_heads * Pmax;
    CUtensorMap mmap;
    if (!encode_tensor_map_2d(&mmap, meta, rows, 2 * D, 64, C::TILE, true)) return GQAQ_ERR_CUDA;
    ScoreParams p;
    p.q = q; p.valid_len = vl; p.scores = scores; p.status = ctx.status;
    p.B = d->batch; p.Hkv = d->num_kv_heads; p.Lmax = d->max_len; p.Pmax = Pmax; p.S = d->page_size;
    p.timeout_ns = ctx.timeout_ns;
    return launch_kernel(kern, dim3(grid), dim3(C::THREADS), C::SMEM, ctx, 0, mmap, p) == cudaSuccess
               ? GQAQ_OK
               : GQAQ_ERR_CUDA;
}

template <int D>
int launch_score_g(const gqaq_dims *d, const __half *q, const __half *meta, const int *vl, float *scores,
                   const LaunchCtx &ctx) {
    switch (d->num_q_heads / d->num_kv_heads) {
        case 1: return launch_score_t<D, 1>(d, q, meta, vl, scores, ctx);
        case 2: return launch_score_t<D, 2>(d, q, meta, vl, scores, ctx);
        case 4: return launch_score_t<D, 4>(d, q, meta, vl, scores, ctx);
        case 8: return launch_score_t<D, 8>(d, q, meta, vl, scores, ctx);
        default: return GQAQ_ERR_UNSUPPORTED;
    }
}
}  // namespace

int launch_append_kv(const gqaq_dims *d, __half *kc, __half *vc, __half *meta, const __half *kn,
                     const __half *vn, const int *pos, const LaunchCtx &ctx) {
    switch (d->head_dim) {
        case 64: return launch_append_t<64>(d, kc, vc, meta, kn, vn, pos, ctx);
        case 128: return launch_append_t<128>(d, kc, vc, meta, kn, vn, pos, ctx);
        default: return GQAQ_ERR_UNSUPPORTED;
    }
}

int launch_update_meta(const gqaq_dims *d, const __half *kc, const int *vl, __half *meta, int p0, int p1,
                       const LaunchCtx &ctx) {
    switch (d->head_dim) {
        case 64: return launch_meta_t<64>(d, kc, vl, meta, p0, p1, ctx);
        case 128: return launch_meta_t<128>(d, kc, vl, meta, p0, p1, ctx);
        default: return GQAQ_ERR_UNSUPPORTED;
    }
}

int launch_score_pages(const gqaq_dims *d, const __half *q, const __half *meta, const int *vl, float *scores,
                       const LaunchCtx &ctx) {
    switch (d->head_dim) {
        case 64: return launch_score_g<64>(d, q, meta, vl, scores, ctx);
        case 128: return launch_score_g<128>(d, q, meta, vl, scores, ctx);
        default: return GQAQ_ERR_UNSUPPORTED;
    }
}

int launch_topk_pages(const gqaq_dims *d, const float *scores, const int *vl, int k, int *page_idx,
                      const LaunchCtx &ctx) {
    static int attr_done[kMaxDevices] = {0};
    const int Pmax = (d->max_len + d->page_size - 1) / d->page_size;
    if (Pmax > kTopkMaxPages) return GQAQ_ERR_UNSUPPORTED;
    const int smem = Pmax * 4;
    if (ctx.device < 0 || ctx.device >= kMaxDevices) return GQAQ_ERR_CUDA;
    if (!attr_done[ctx.device]) {
        if (cudaFuncSetAttribute(topk_pages_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kTopkMaxPages * 4) != cudaSuccess)
            return GQAQ_ERR_CUDA;
        attr_done[ctx.device] = 1;
    }
    TopkParams p;
    p.scores = scores; p.valid_len = vl; p.page_idx = page_idx; p.status = ctx.status;
    p.B = d->batch; p.Hkv = d->num_kv_heads; p.Lmax = d->max_len; p.Pmax = Pmax; p.S = d->page_size;
    p.k = k;
    return launch_kernel(topk_pages_kernel, dim3(d->num_kv_heads, d->batch), dim3(kTopkThreads), smem, ctx, 0, p) ==
                   cudaSuccess
               ? GQAQ_OK
               : GQAQ_ERR_CUDA;
}

}  // namespace gqaq
