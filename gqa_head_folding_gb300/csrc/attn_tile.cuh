// attn_tile.cuh -- the per-warp decode-attention tile shared by the
// split-context kernel (attn.cu) and the fused Quest kernel (quest_fused.cu).
//
// "Core ML Decode Optimization: Removing the 1.9 GiB Per-Token Copy Caused by
// GQA repeat_kv", section 3: the G query rows that share a KV head form one
// [G, D] block, so each K and V row staged in shared memory serves all G rows.
// Scale, mask and softmax act per row along the context axis, so every row
// keeps its own running max m, sum l and accumulator.
//
// Stage layout (filled by TMA): K as D/64 column blocks of [128 rows][128 B]
// with the 128-byte swizzle (16-byte chunk c of row r sits at chunk c ^ (r & 7)),
// then V as [128 rows][D] halves. Consumer warp w owns rows 16w .. 16w+15.
//
// Per 16-token sub-tile a warp:
//  1. q.k: 4 lanes share a token (lane = 8*part + jt handles tokens jt and jt+8),
//     each lane covering D/4 channels with fp16 x fp16 -> fp32 FMAs (products
//     are exact in fp32);
//  2. reduce-scatters the 4 partial dots so a lane ends up owning the full dot
//     of G/4 query rows (rows are duplicated over lanes when G < 4);
//  3. runs the online softmax (log2 domain) for the rows it owns, stores p to
//     shared memory pair-interleaved ([token/2][row][2]) and broadcasts each
//     row's rescale factor;
//  4. accumulates p @ V over token pairs with packed f32x2 FMAs: lane l owns
//     channels [l*D/32, (l+1)*D/32) of every row, with separate even-token and
//     odd-token sums.
#pragma once

#include "common.cuh"

namespace gqaq {

template <int D, int G>
struct TileCfg {
    static constexpr int NCW = 8;                 // consumer warps per CTA
    static constexpr int TILE = 128;              // tokens per stage (8 pages of 16)
    static constexpr int SUB = 16;                // tokens per consumer warp
    static constexpr int KH = D / 64;             // 128-byte column blocks per K row
    static constexpr int KBLK = TILE * 128;       // bytes of one K column block
    static constexpr int KBYTES = KH * KBLK;      // = TILE * D * 2
    static constexpr int VBYTES = TILE * D * 2;
    static constexpr int STAGE = KBYTES + VBYTES;
    static constexpr int LPT = 4;                 // lanes per token in q.k
    static constexpr int TPP = 8;                 // tokens per lane pass
    static constexpr int NTL = 2;                 // tokens per lane
    static constexpr int DQ = D / LPT;            // channels per lane in q.k
    static constexpr int NCH = DQ / 8;            // 16-byte chunks per lane in q.k
    static constexpr int DPL = D / 32;            // channels per lane in p @ V
    static constexpr bool QREG = (G * D <= 512);  // q block held in registers
    static constexpr int GQ = QREG ? G : 4;       // query rows per q.k pass
    static constexpr int NPASS = G / GQ;
    static constexpr int HPL = G >= 4 ? G / 4 : 1;  // softmax rows owned per lane
    static constexpr int QBYTES = G * D * 2;
    static constexpr int PBYTES = NCW * SUB * G * 4;
    static constexpr int MERGE = NCW * G * (D + 2) * 4;
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "group");
};

// Two E4M3 codes (low byte = first element) -> fp16x2 (low half = first).
// Every E4M3 value is exactly representable in fp16.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    uint32_t r;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(r) : "r"(two));
    return r;
}

// Four E4M3 codes (byte 0 first) -> two fp16x2: lo holds bytes 0, 1 and hi
// bytes 2, 3. The word is split into its 16-bit halves as registers, so no
// mask or shift is spent on either half.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// K layout in a stage: KPAGE = false: KH column blocks of TILE rows x 128 B
// ([kh][row]); KPAGE = true: row after row, each row's KH 128-byte blocks
// side by side ([row][kh]), as one 3-D TMA box per page writes them. Both
// are 128-byte swizzled: 16-byte chunk c of 128-byte line L sits at c ^ (L & 7).
// KV8 = true: K and V hold E4M3 codes, one byte per channel. K rows are D
// bytes: D = 128 rows are 128-byte swizzled like above (chunk c of row r at
// c ^ (r & 7)); D = 64 rows are 64-byte swizzled (chunk c of row r at
// c ^ ((r >> 1) & 3)). V rows are D bytes, not swizzled. Products of the fp16
// q with the decoded codes are exact; the caller folds the per-tensor K scale
// into scale_log2 and multiplies the output by the V scale.
template <int D, int G, bool KPAGE = false, bool KV8 = false>
struct WarpAttn {
    using C = TileCfg<D, G>;
    static_assert(!(KPAGE && KV8), "8-bit K is dense-only");
    int lane, part, jt, cw;
    uint32_t krow_off, kx0, pbw;
    uint4 qr[C::GQ][C::NCH];
    float m[C::HPL], l[C::HPL];
    float2 acc[G][C::DPL];

    __device__ __forceinline__ void init(int warp, int lane_, uint32_t pbuf_base) {
        lane = lane_;
        cw = warp;
        part = lane >> 3;
        jt = lane & 7;
        const int c0 = part * C::DQ;
        if (KV8) {
            const int row = cw * C::SUB + jt;
            krow_off = (uint32_t)(row * D);
            kx0 = (D == 128) ? (uint32_t)((2 * part) ^ jt) : (uint32_t)(part ^ ((jt >> 1) & 3));
        } else if (KPAGE) {
            const int line = (cw * C::SUB + jt) * C::KH + c0 / 64;
            krow_off = (uint32_t)(line * 128);
            kx0 = (uint32_t)(((c0 % 64) / 8) ^ (line & 7));  // rows jt and jt+8: same (line & 7)
        } else {
            krow_off = (uint32_t)((c0 / 64) * C::KBLK + (cw * C::SUB + jt) * 128);
            kx0 = (uint32_t)(((c0 % 64) / 8) ^ jt);  // rows jt and jt+8 share (row & 7)
        }
        pbw = pbuf_base + (uint32_t)(cw * C::SUB * G * 4);
    }
    // Row of the query group whose softmax this lane owns (i < HPL).
    __device__ __forceinline__ int row(int i) const { return (part * G) / 4 + i; }
    // First lane part that owns row g.
    static __device__ __forceinline__ int owner_part(int g) { return G >= 4 ? g / (G / 4) : (g * 4) / G; }
    // Lanes whose softmax state counts (one lane part per row when G < 4).
    __device__ __forceinline__ bool primary() const { return G >= 4 || (part % (G >= 4 ? 1 : 4 / G)) == 0; }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int i = 0; i < C::HPL; ++i) {
            m[i] = -INFINITY;
            l[i] = 0.f;
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < C::DPL; ++e) acc[g][e] = make_float2(0.f, 0.f);
    }

    // q rows of one unit, this lane's D/4 channels (register-resident case).
    __device__ __forceinline__ void load_q(const __half *qg) {
        if (C::QREG) {
#pragma unroll
            for (int g = 0; g < C::GQ; ++g)
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    qr[g][c] = *reinterpret_cast<const uint4 *>(qg + g * D + part * C::DQ + c * 8);
        }
    }

    __device__ __forceinline__ void reduce_scatter(const float (&a)[G], float (&s)[C::HPL]) const {
        const bool b1 = (lane >> 4) & 1, b0 = (lane >> 3) & 1;
        if constexpr (G == 1) {
            float x = a[0];
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            s[0] = x;
        } else if constexpr (G == 2) {
            const float send = b1 ? a[0] : a[G - 1], keep = b1 ? a[G - 1] : a[0];
            float y = keep + __shfl_xor_sync(0xffffffffu, send, 16);
            y += __shfl_xor_sync(0xffffffffu, y, 8);
            s[0] = y;
        } else {
            constexpr int H = G / 2;  // rows kept after the first exchange
            float w[H];
#pragma unroll
            for (int k = 0; k < H; ++k) {
                const float send = b1 ? a[k] : a[k + H], keep = b1 ? a[k + H] : a[k];
                w[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
            }
#pragma unroll
            for (int k = 0; k < C::HPL; ++k) {
                const float send = b0 ? w[k] : w[k + C::HPL], keep = b0 ? w[k + C::HPL] : w[k];
                s[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
            }
        }
    }

    // One 16-token sub-tile. kbase/vbase: shared addresses of the stage's K and
    // V; nvalid: valid tokens (a prefix) of this warp's 16 rows, 1..16.
    __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int nvalid, float scale_log2,
                                         const __half *q_s) {
        // ---- 1. partial dots over this lane's D/4 channels ----
        float a[C::NTL][G];
#pragma unroll
        for (int pass = 0; pass < C::NPASS; ++pass) {
            if (!C::QREG) {
#pragma unroll
                for (int g = 0; g < C::GQ; ++g)
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c)
                        qr[g][c] = lds128(smem_u32(q_s + (pass * C::GQ + g) * D + part * C::DQ + c * 8));
            }
#pragma unroll
            for (int u = 0; u < C::NTL; ++u) {
                float a0[C::GQ], a1[C::GQ];
#pragma unroll
                for (int g = 0; g < C::GQ; ++g) a0[g] = a1[g] = 0.f;
                const uint32_t kro = KV8 ? kbase + krow_off + (uint32_t)(u * C::TPP * D)
                                         : kbase + krow_off + (uint32_t)(u * C::TPP * (KPAGE ? C::KH : 1) * 128);
                uint4 k8 = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c) {
                    uint4 kc;
                    if (KV8) {  // one 16-byte chunk of codes feeds two fp16 chunks of q
                        if ((c & 1) == 0) k8 = lds128(kro + ((kx0 ^ (uint32_t)(c >> 1)) << 4));
                        const uint32_t lo = (c & 1) ? k8.z : k8.x, hi = (c & 1) ? k8.w : k8.y;
                        e4m3x4_to_f16x2x2(lo, kc.x, kc.y);
                        e4m3x4_to_f16x2x2(hi, kc.z, kc.w);
                    } else {
                        kc = lds128(kro + ((kx0 ^ (uint32_t)c) << 4));
                    }
#pragma unroll
                    for (int g = 0; g < C::GQ; ++g) {
                        a0[g] = fma_h_lo(qr[g][c].x, kc.x, a0[g]);
                        a1[g] = fma_h_hi(qr[g][c].x, kc.x, a1[g]);
                        a0[g] = fma_h_lo(qr[g][c].y, kc.y, a0[g]);
                        a1[g] = fma_h_hi(qr[g][c].y, kc.y, a1[g]);
                        a0[g] = fma_h_lo(qr[g][c].z, kc.z, a0[g]);
                        a1[g] = fma_h_hi(qr[g][c].z, kc.z, a1[g]);
                        a0[g] = fma_h_lo(qr[g][c].w, kc.w, a0[g]);
                        a1[g] = fma_h_hi(qr[g][c].w, kc.w, a1[g]);
                    }
                }
#pragma unroll
                for (int g = 0; g < C::GQ; ++g) a[u][pass * C::GQ + g] = a0[g] + a1[g];
            }
        }
        // ---- 2. full dots of the rows this lane owns ----
        float s[C::NTL][C::HPL];
#pragma unroll
        for (int u = 0; u < C::NTL; ++u) reduce_scatter(a[u], s[u]);
        // ---- 3. online softmax (log2 domain) over the 16 tokens ----
        float alpha[C::HPL];
#pragma unroll
        for (int i = 0; i < C::HPL; ++i) {
            float x[C::NTL];
            float tmax = -INFINITY;
#pragma unroll
            for (int u = 0; u < C::NTL; ++u) {
                x[u] = (jt + u * C::TPP < nvalid) ? s[u][i] * scale_log2 : -INFINITY;
                tmax = fmaxf(tmax, x[u]);
            }
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
            const float mnew = fmaxf(m[i], tmax);
            alpha[i] = fast_exp2(m[i] - mnew);
            m[i] = mnew;
            float psum = 0.f;
#pragma unroll
            for (int u = 0; u < C::NTL; ++u) {
                const float pu = fast_exp2(x[u] - mnew);
                psum += pu;
                if (primary()) {
                    const int t = jt + u * C::TPP;
                    asm volatile("st.shared.f32 [%0], %1;" ::"r"(pbw + (uint32_t)((((t >> 1) * G + row(i)) * 2 + (t & 1)) * 4)),
                                 "f"(pu));
                }
            }
            l[i] = l[i] * alpha[i] + psum;
        }
        // ---- 4. rescale every row's accumulator ----
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float al = __shfl_sync(0xffffffffu, alpha[g % C::HPL], owner_part(g) * 8);
#pragma unroll
            for (int e = 0; e < C::DPL; ++e) acc[g][e] = __fmul2_rn(acc[g][e], make_float2(al, al));
        }
        __syncwarp();
        // ---- 5. acc += p @ V, two tokens per packed FMA ----
        const int npairs = (nvalid + 1) >> 1;
        const uint32_t vrow = KV8 ? vbase + (uint32_t)(cw * C::SUB * D + lane * C::DPL)
                                  : vbase + (uint32_t)(cw * C::SUB * D * 2 + lane * C::DPL * 2);
#pragma unroll 1
        for (int jp = 0; jp < npairs; ++jp) {
            const bool has1 = 2 * jp + 1 < nvalid;
            float v0[C::DPL], v1[C::DPL];
            if constexpr (KV8 && D == 128) {  // 4 codes per lane per row
                const uint32_t r0 = lds32(vrow + (uint32_t)(2 * jp * D));
                const uint32_t r1 = has1 ? lds32(vrow + (uint32_t)((2 * jp + 1) * D)) : 0u;
                uint32_t h0, h1, h2, h3;
                e4m3x4_to_f16x2x2(r0, h0, h1);
                e4m3x4_to_f16x2x2(r1, h2, h3);
                const float2 a0 = half2_bits_to_float2(h0);
                const float2 a1 = half2_bits_to_float2(h1);
                const float2 b0 = half2_bits_to_float2(h2);
                const float2 b1 = half2_bits_to_float2(h3);
                v0[0] = a0.x; v0[1] = a0.y; v0[C::DPL > 2 ? 2 : 0] = a1.x; v0[C::DPL > 3 ? 3 : 0] = a1.y;
                v1[0] = b0.x; v1[1] = b0.y; v1[C::DPL > 2 ? 2 : 0] = b1.x; v1[C::DPL > 3 ? 3 : 0] = b1.y;
            } else if constexpr (KV8) {  // D = 64: 2 codes per lane per row
                uint32_t r0, r1 = 0u;
                asm volatile("ld.shared.u16 %0, [%1];" : "=r"(r0) : "r"(vrow + (uint32_t)(2 * jp * D)));
                if (has1) asm volatile("ld.shared.u16 %0, [%1];" : "=r"(r1) : "r"(vrow + (uint32_t)((2 * jp + 1) * D)));
                const float2 a = half2_bits_to_float2(e4m3x2_to_f16x2(r0));
                const float2 b = half2_bits_to_float2(e4m3x2_to_f16x2(r1));
                v0[0] = a.x; v0[C::DPL > 1 ? 1 : 0] = a.y;
                v1[0] = b.x; v1[C::DPL > 1 ? 1 : 0] = b.y;
            } else if constexpr (D == 128) {
                const uint2 r0 = lds64(vrow + (uint32_t)(2 * jp * D * 2));
                uint2 r1 = lds64(vrow + (uint32_t)((2 * jp + 1) * D * 2));
                if (!has1) r1 = make_uint2(0u, 0u);
                const float2 f00 = half2_bits_to_float2(r0.x), f01 = half2_bits_to_float2(r0.y);
                const float2 f10 = half2_bits_to_float2(r1.x), f11 = half2_bits_to_float2(r1.y);
                v0[0] = f00.x; v0[1] = f00.y; v0[C::DPL > 2 ? 2 : 0] = f01.x; v0[C::DPL > 3 ? 3 : 0] = f01.y;
                v1[0] = f10.x; v1[1] = f10.y; v1[C::DPL > 2 ? 2 : 0] = f11.x; v1[C::DPL > 3 ? 3 : 0] = f11.y;
            } else {
                const uint32_t r0 = lds32(vrow + (uint32_t)(2 * jp * D * 2));
                uint32_t r1 = lds32(vrow + (uint32_t)((2 * jp + 1) * D * 2));
                if (!has1) r1 = 0u;
                const float2 f0 = half2_bits_to_float2(r0), f1 = half2_bits_to_float2(r1);
                v0[0] = f0.x; v0[C::DPL > 1 ? 1 : 0] = f0.y;
                v1[0] = f1.x; v1[C::DPL > 1 ? 1 : 0] = f1.y;
            }
            float2 pp[G];
            const uint32_t pa = pbw + (uint32_t)(jp * G * 8);
            if constexpr (G >= 2) {
#pragma unroll
                for (int g = 0; g < G; g += 2) {
                    const uint4 x = lds128(pa + (uint32_t)(g * 8));
                    pp[g] = make_float2(__uint_as_float(x.x), __uint_as_float(x.y));
                    pp[g + 1 < G ? g + 1 : g] = make_float2(__uint_as_float(x.z), __uint_as_float(x.w));
                }
            } else {
                const uint2 x = lds64(pa);
                pp[0] = make_float2(__uint_as_float(x.x), __uint_as_float(x.y));
            }
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < C::DPL; ++e) acc[g][e] = __ffma2_rn(pp[g], make_float2(v0[e], v1[e]), acc[g][e]);
        }
    }

    // Write this warp's state to its slot of the merge buffer [NCW][G][D+2]:
    // (m, l, acc[D]) per row; l is summed over the 8 token lanes first.
    __device__ __forceinline__ void store_state(float *merge) {
        float *mw = merge + cw * G * (D + 2);
#pragma unroll
        for (int i = 0; i < C::HPL; ++i) {
            float x = l[i];
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            if (jt == 0 && primary()) {
                mw[row(i) * (D + 2)] = m[i];
                mw[row(i) * (D + 2) + 1] = x;
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < C::DPL; ++e) mw[g * (D + 2) + 2 + lane * C::DPL + e] = acc[g][e].x + acc[g][e].y;
    }
};

// Merge the 8 warp states of a CTA, element (g, d) of the G x D block:
// m* = max_w m_w, l* = sum_w 2^(m_w - m*) l_w, a* = sum_w 2^(m_w - m*) acc_w.
// Pages gathered into a 128-row stage, page size S in {8, 16, 32, 64}. Each
// page takes a slot of max(S, 16) rows (one TMA box of S rows at the slot's
// start), so a stage holds 128 / max(S, 16) pages. Consumer warp w owns rows
// 16w .. 16w+15: they lie in page (16w) / slot, from row (16w) % slot, and
// its valid rows are a prefix (only a sequence's last page can be partial).
struct PageSlots {
    int S, slot, ppt;
    __device__ __forceinline__ void init(int page_size) {
        S = page_size;
        slot = page_size > 16 ? page_size : 16;
        ppt = 128 / slot;
    }
    __device__ __forceinline__ int warp_page(int w) const { return (16 * w) / slot; }
    // Valid rows of warp w when its page `page` (a valid page) of a sequence of
    // `len` tokens is loaded.
    __device__ __forceinline__ int warp_rows(int w, int page, int len) const {
        int rows = len - page * S;
        rows = rows < S ? rows : S;
        const int r = rows - (16 * w) % slot;
        return r < 0 ? 0 : (r < 16 ? r : 16);
    }
};

template <int D, int G>
__device__ __forceinline__ void merge_warps(const float *merge, int g, int d, float &mst, float &ls, float &as) {
    constexpr int NCW = TileCfg<D, G>::NCW;
    mst = -INFINITY;
#pragma unroll
    for (int w = 0; w < NCW; ++w) mst = fmaxf(mst, merge[(w * G + g) * (D + 2)]);
    ls = 0.f;
    as = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
        const float *st = merge + (w * G + g) * (D + 2);
        if (st[0] != -INFINITY) {
            const float f = fast_exp2(st[0] - mst);
            ls += f * st[1];
            as += f * st[2 + d];
        }
    }
}

}  // namespace gqaq
