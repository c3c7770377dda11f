// attn_mma.cuh -- one consumer warp's share of a decode-attention tile on the
// tensor cores (mma.sync m16n8k16, fp16 operands, fp32 accumulation).
//
// "Core ML Decode Optimization ...", section 3 ("Fold Q Instead of Expanding
// KV"): the G query rows of one KV head form a [G, D] block that meets every
// K and V row once. With G <= 8 that block is the N = 8 side of the MMA, and
// the 16 tokens a warp owns are the M = 16 side, so both products of a tile
// are tensor-core contractions with no copy of K or V:
//   S^T [16 tokens x 8 rows] = K [16 x D] . Q^T [D x 8]          (D/16 MMAs)
//   O^T [D x 8 rows]        += V^T [D x 16 tokens] . P^T [16 x 8] (D/16 MMAs)
// Softmax runs in the log2 domain on the S^T fragments (each lane holds two
// query columns of two tokens) against a lazy reference max: the column max
// is gathered across lanes, and l and O rescaled, only when a tile holds a
// score more than 2^8 above the reference, so P <= 256. P is rounded to fp16
// once and turned into the B operand of the second product with
// movmatrix.trans. Rows G..7 of the N side are zero queries whose results are
// never stored.
//
// fp16 caches: K and V stages share one layout, KH column blocks of 128-byte
// lines, 128-byte swizzled (dense: [kh][row] blocks of TILE lines; KPAGE:
// [row][kh], as the page-major 3-D box writes them). ldmatrix brings K
// fragments and, transposed, V^T fragments.
// E4M3 caches (KV8): rows of D bytes, swizzled by 128 bytes (D = 128) or 64
// bytes (D = 64). A lane reads its K bytes as whole 16-byte chunks and
// decodes them into fragments; the channel order inside the contraction is
// permuted to match (q uses the same permutation, so q.k is unchanged). V^T
// fragments pair two tokens' codes with a byte permute before decoding.
// INT4 caches (KV4): rows of D/2 bytes (channel 2i in the low nibble of byte
// i) plus one fp32 scale per token row. Nibbles decode exactly to fp16 (the
// 1024 + n bit trick, minus 1032; the high nibble of a byte in place, as
// 1024 + 16 n, then one fma), one shift per word; the K scale multiplies the token's fp32
// score and the V scale its probability, so both contractions run on the
// integer levels. The channel order is permuted as for E4M3.
#pragma once

#include "attn_tile.cuh"

namespace gqaq {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t r;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

// d += a (16x16, row) . b (16x8, col), fp16 in, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two fp32 -> fp16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t byte_perm(uint32_t x, uint32_t y, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(y), "r"(sel));
    return r;
}

// The nibbles at bits 0 and 16 of x -> fp16x2 of (nibble - 8), exact: OR-ing a
// nibble n into the mantissa of 1024.0 gives 1024 + n, less 1032.
__device__ __forceinline__ uint32_t nib2_lo_f16x2(uint32_t x) {
    uint32_t t, r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(t) : "r"(x), "r"(0x000F000Fu), "r"(0x64006400u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(0x64086408u));  // - (1024 + 8)
    return r;
}
// The nibbles at bits 4 and 20 of x, without a shift: in place they give
// 1024 + 16 n, and (1024 + 16 n) / 16 - 72 = n - 8 is one exact fma.
__device__ __forceinline__ uint32_t nib2_hi_f16x2(uint32_t x) {
    uint32_t t, r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(t) : "r"(x), "r"(0x00F000F0u), "r"(0x64006400u));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(t), "r"(0x2C002C00u), "r"(0xD480D480u));  // x/16 - 72
    return r;
}

template <int D, int G, bool KPAGE = false, int KV = 0>
struct MmaAttn {
    using C = TileCfg<D, G>;
    static constexpr bool KV8 = KV == 1;  // E4M3 codes
    static constexpr bool KV4 = KV == 2;  // INT4 levels + per-token scales
    static_assert(!(KPAGE && KV != 0), "8-bit and 4-bit stages are dense-only");
    static constexpr bool QREG = true;   // q fragments live in registers
    static constexpr int KS = D / 16;    // k-steps of q.k, m-blocks of p @ V
    int lane, cw, r, c;                  // r = lane / 4 (token / channel row), c = lane % 4 (column pair)
    uint32_t qb[KS][2];                  // B fragments of Q^T
    float m[2], l[2];                    // columns 2c, 2c+1: running max (log2 domain), partial sum
    float o[KS][4];                      // O^T fragments

    // ---- shared-memory addressing ----
    // fp16 stage: byte address of the 16-byte chunk (row, ch8) (8 channels).
    __device__ __forceinline__ static uint32_t chunk16(uint32_t base, int row, int ch8) {
        const int kh = ch8 >> 3, cc = ch8 & 7;
        if (KPAGE) {
            const int line = row * C::KH + kh;
            return base + (uint32_t)(line * 128 + ((cc ^ (line & 7)) << 4));
        }
        return base + (uint32_t)(kh * C::KBLK + row * 128 + ((cc ^ (row & 7)) << 4));
    }
    // INT4 stage: codes [TILE][D/2] unswizzled, then the TILE fp32 scales.
    static constexpr int CODE4 = C::TILE * D / 2;
    // E4M3 stage: byte address of logical byte `byte` (a multiple of 8) of row `row`.
    __device__ __forceinline__ static uint32_t byte8(uint32_t base, int row, int byte) {
        if (D == 128) return base + (uint32_t)(row * 128 + ((((byte >> 4) ^ (row & 7))) << 4) + (byte & 15));
        return base + (uint32_t)(row * 64 + ((((byte >> 4) ^ ((row >> 1) & 3))) << 4) + (byte & 15));
    }

    __device__ __forceinline__ void init(int warp, int lane_, uint32_t /*pbuf_base*/) {
        lane = lane_;
        cw = warp;
        r = lane >> 2;
        c = lane & 3;
    }

    __device__ __forceinline__ void reset() {
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
#pragma unroll
        for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    }

    // B fragments of Q^T for the unit's [G][D] block (row n = r; rows >= G are zero).
    // fp16 stages: k-step j covers channels 16j .. 16j+15 in natural order.
    // E4M3 stages: k-step j of column pair c covers channels (D/4) c + 4j .. +3.
    // INT4 stages: k-step j of column pair c covers base, base+4 (b0) and
    // base+1, base+5 (b1), base = (D/4) c + 8 (j/2) + 2 (j%2).
    __device__ __forceinline__ void load_q(const __half *qg) {
        const bool live = r < G;
        const __half *qrow = qg + (live ? r : 0) * D;
        const uint16_t *qh = reinterpret_cast<const uint16_t *>(qrow);
#pragma unroll
        for (int j = 0; j < KS; ++j) {
            if (KV4) {
                const int base = (D / 4) * c + 8 * (j >> 1) + 2 * (j & 1);
                qb[j][0] = live ? ((uint32_t)qh[base] | ((uint32_t)qh[base + 4] << 16)) : 0u;
                qb[j][1] = live ? ((uint32_t)qh[base + 1] | ((uint32_t)qh[base + 5] << 16)) : 0u;
            } else if (KV8) {
                const uint2 x = live ? *reinterpret_cast<const uint2 *>(qrow + (D / 4) * c + 4 * j) : make_uint2(0u, 0u);
                qb[j][0] = x.x;
                qb[j][1] = x.y;
            } else {
                qb[j][0] = live ? *reinterpret_cast<const uint32_t *>(qrow + 16 * j + 2 * c) : 0u;
                qb[j][1] = live ? *reinterpret_cast<const uint32_t *>(qrow + 16 * j + 8 + 2 * c) : 0u;
            }
        }
    }

    // ---- S^T of the 16 stage rows row0 .. row0+15 (K scales applied for INT4) ----
    __device__ __forceinline__ void qk(uint32_t kbase, int row0, float (&s)[4]) const {
        s[0] = s[1] = s[2] = s[3] = 0.f;
        if constexpr (KV4) {
            constexpr int NW = D / 32;  // words of a row this lane decodes (D/4 channels)
            uint32_t wa[NW], wb[NW];
            const uint32_t ra = kbase + (uint32_t)((row0 + r) * (D / 2) + (D / 8) * c);
            const uint32_t rb = ra + (uint32_t)(8 * (D / 2));
            if constexpr (NW == 2) {
                const uint2 x = lds64(ra), y = lds64(rb);
                wa[0] = x.x; wa[NW - 1] = x.y; wb[0] = y.x; wb[NW - 1] = y.y;
            } else {
                const uint4 x = lds128(ra), y = lds128(rb);
                wa[0] = x.x; wa[1 % NW] = x.y; wa[2 % NW] = x.z; wa[3 % NW] = x.w;
                wb[0] = y.x; wb[1 % NW] = y.y; wb[2 % NW] = y.z; wb[3 % NW] = y.w;
            }
#pragma unroll
            for (int j = 0; j < KS; ++j) {
                const int e = 2 * (j & 1);
                const uint32_t xa = wa[j >> 1] >> (4 * e), xb = wb[j >> 1] >> (4 * e);  // nibble pairs at bits 4e, 4e + 4
                uint32_t a[4];
                a[0] = nib2_lo_f16x2(xa);
                a[1] = nib2_lo_f16x2(xb);
                a[2] = nib2_hi_f16x2(xa);
                a[3] = nib2_hi_f16x2(xb);
                mma_16816(s, a, qb[j][0], qb[j][1]);
            }
            const float ks0 = __uint_as_float(lds32(kbase + (uint32_t)(CODE4 + (row0 + r) * 4)));
            const float ks1 = __uint_as_float(lds32(kbase + (uint32_t)(CODE4 + (row0 + r + 8) * 4)));
            s[0] *= ks0;
            s[1] *= ks0;
            s[2] *= ks1;
            s[3] *= ks1;
        } else if (KV8) {
            constexpr int BPL = D / 4;  // bytes of a row this lane decodes
            uint4 ka[BPL / 16], kb[BPL / 16];
#pragma unroll
            for (int h = 0; h < BPL / 16; ++h) {
                ka[h] = lds128(byte8(kbase, row0 + r, BPL * c + 16 * h));
                kb[h] = lds128(byte8(kbase, row0 + r + 8, BPL * c + 16 * h));
            }
#pragma unroll
            for (int j = 0; j < KS; ++j) {
                const uint4 &xa = ka[j >> 2], &xb = kb[j >> 2];
                const uint32_t wa = (j & 3) == 0 ? xa.x : (j & 3) == 1 ? xa.y : (j & 3) == 2 ? xa.z : xa.w;
                const uint32_t wb = (j & 3) == 0 ? xb.x : (j & 3) == 1 ? xb.y : (j & 3) == 2 ? xb.z : xb.w;
                uint32_t a[4];
                e4m3x4_to_f16x2x2(wa, a[0], a[2]);
                e4m3x4_to_f16x2x2(wb, a[1], a[3]);
                mma_16816(s, a, qb[j][0], qb[j][1]);
            }
        } else {
            const int mi = lane >> 3, rr = lane & 7;
            const int krow = row0 + (mi & 1) * 8 + rr;
#pragma unroll
            for (int j = 0; j < KS; ++j) {
                uint32_t a[4];
                ldsm_x4(chunk16(kbase, krow, 2 * j + (mi >> 1)), a);
                mma_16816(s, a, qb[j][0], qb[j][1]);
            }
        }
    }

    // ---- O^T += V^T . P^T over the 16 stage rows row0 .. row0+15 ----
    // Rows past the valid prefix may hold anything (even NaN codes): with
    // `partial` their V^T entries are zeroed by mk0 / mk1, since 0 * NaN
    // would poison the sum.
    __device__ __forceinline__ void pv(uint32_t vbase, int row0, uint32_t pb0, uint32_t pb1, bool partial,
                                       uint32_t mk0, uint32_t mk1) {
        if constexpr (KV4) {
            constexpr int NW = D / 64;  // words of a token row this lane reads (channels (D/8) r ..)
            uint32_t w[4][NW];          // tokens 2c, 2c+1, 2c+8, 2c+9
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int row = row0 + 2 * c + (t & 1) + (t >> 1) * 8;
                const uint32_t addr = vbase + (uint32_t)(row * (D / 2) + (D / 16) * r);
                if constexpr (NW == 2) {
                    const uint2 v = lds64(addr);
                    w[t][0] = v.x;
                    w[t][NW - 1] = v.y;
                } else {
                    w[t][0] = lds32(addr);
                }
            }
#pragma unroll
            for (int i = 0; i < KS; ++i) {
                // m-block i: row r <-> channel (D/8) r + 2i, row r + 8 <-> (D/8) r + 2i + 1
                const int wd = i >> 2, k = 2 * (i & 3);            // channel k, k+1 of word wd
                const uint32_t sel = k < 4 ? 0x5410u : 0x7632u;      // bytes holding channels 0-3 / 4-7
                const int sh = 4 * (k & 3);
                const uint32_t lo = byte_perm(w[0][wd], w[1][wd], sel);  // tokens 2c | 2c+1
                const uint32_t hi = byte_perm(w[2][wd], w[3][wd], sel);  // tokens 2c+8 | 2c+9
                const uint32_t xl = lo >> sh, xh = hi >> sh;  // channel k at bits 0 / 16, k + 1 at 4 / 20
                uint32_t a[4];
                a[0] = nib2_lo_f16x2(xl);
                a[1] = nib2_hi_f16x2(xl);
                a[2] = nib2_lo_f16x2(xh);
                a[3] = nib2_hi_f16x2(xh);
                if (partial) mask_tokens(a, mk0, mk1);
                mma_16816(o[i], a, pb0, pb1);
            }
        } else if (KV8) {
            constexpr int BPL = D / 8;  // bytes of a token row this lane reads (channels BPL r ..)
            uint32_t w[4][BPL / 4];     // tokens 2c, 2c+1, 2c+8, 2c+9
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int row = row0 + 2 * c + (t & 1) + (t >> 1) * 8;
                if constexpr (BPL == 16) {
                    const uint4 v = lds128(byte8(vbase, row, BPL * r));
                    w[t][0] = v.x;
                    w[t][1] = v.y;
                    w[t][2 % (BPL / 4)] = v.z;
                    w[t][3 % (BPL / 4)] = v.w;
                } else {
                    const uint2 v = lds64(byte8(vbase, row, BPL * r));
                    w[t][0] = v.x;
                    w[t][1 % (BPL / 4)] = v.y;
                }
            }
#pragma unroll
            for (int i = 0; i < KS; ++i) {
                // m-block i: row r <-> channel BPL r + 2i, row r + 8 <-> BPL r + 2i + 1
                const int wd = i >> 1;
                const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
                const uint32_t lo = byte_perm(w[0][wd], w[1][wd], sel);  // tokens 2c, 2c+1
                const uint32_t hi = byte_perm(w[2][wd], w[3][wd], sel);  // tokens 2c+8, 2c+9
                uint32_t a[4];
                e4m3x4_to_f16x2x2(lo, a[0], a[1]);
                e4m3x4_to_f16x2x2(hi, a[2], a[3]);
                if (partial) mask_tokens(a, mk0, mk1);
                mma_16816(o[i], a, pb0, pb1);
            }
        } else {
            const int mi = lane >> 3, rr = lane & 7;
            const int vrow = row0 + (mi >> 1) * 8 + rr;
#pragma unroll
            for (int i = 0; i < KS; ++i) {
                uint32_t a[4];
                ldsm_x4_trans(chunk16(vbase, vrow, 2 * i + (mi & 1)), a);
                if (partial) mask_tokens(a, mk0, mk1);
                mma_16816(o[i], a, pb0, pb1);
            }
        }
    }

    // NS sub-tiles of 16 stage rows each, from row0 (a multiple of 16), with
    // one online-softmax step over all 16 NS tokens. kbase/vbase: shared
    // addresses of the stage's K and V; nv[h]: valid tokens (a prefix) of
    // sub-tile h, 0..16, at least one of them nonzero. The sub-tiles' MMA
    // chains are independent, so the scheduler overlaps them.
    template <int NS>
    __device__ __forceinline__ void tile_n(uint32_t kbase, uint32_t vbase, int row0, const int (&nv)[NS],
                                           float scale_log2) {
        // ---- 1. S^T = K . Q^T per sub-tile ----
        float s[NS][4];
#pragma unroll
        for (int h = 0; h < NS; ++h) qk(kbase, row0 + 16 * h, s[h]);
        // ---- 2. online softmax per query column (log2 domain), lazy reference max ----
        // s[h][0], s[h][1]: token r of sub-tile h, columns 2c, 2c+1; s[h][2], s[h][3]: token r + 8.
        // m is a reference max shared by the 8 lanes of a column pair; it moves (with
        // the rescale of l and O) only when some score exceeds it by more than 2^8,
        // so every P = 2^(s - m) stays at most 256 and fp16 keeps its precision.
        bool v0[NS], v1[NS];
        float t0 = -INFINITY, t1 = -INFINITY;
#pragma unroll
        for (int h = 0; h < NS; ++h) {
            v0[h] = r < nv[h];
            v1[h] = r + 8 < nv[h];
            s[h][0] *= scale_log2;
            s[h][1] *= scale_log2;
            s[h][2] *= scale_log2;
            s[h][3] *= scale_log2;
            if (nv[h] < C::SUB) {  // warp-uniform: a sub-tile with rows past the valid prefix
                s[h][0] = v0[h] ? s[h][0] : -INFINITY;
                s[h][1] = v0[h] ? s[h][1] : -INFINITY;
                s[h][2] = v1[h] ? s[h][2] : -INFINITY;
                s[h][3] = v1[h] ? s[h][3] : -INFINITY;
            }
            t0 = fmaxf(t0, fmaxf(s[h][0], s[h][2]));
            t1 = fmaxf(t1, fmaxf(s[h][1], s[h][3]));
        }
        if (__any_sync(0xffffffffu, t0 > m[0] + 8.f || t1 > m[1] + 8.f)) {
#pragma unroll
            for (int o_ = 4; o_ < 32; o_ <<= 1) {
                t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, o_));
                t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, o_));
            }
            const float mn0 = fmaxf(m[0], t0), mn1 = fmaxf(m[1], t1);  // some token is valid: finite
            const float al0 = fast_exp2(m[0] - mn0), al1 = fast_exp2(m[1] - mn1);
            m[0] = mn0;
            m[1] = mn1;
            l[0] *= al0;
            l[1] *= al1;
#pragma unroll
            for (int i = 0; i < KS; ++i) {
                o[i][0] *= al0;
                o[i][1] *= al1;
                o[i][2] *= al0;
                o[i][3] *= al1;
            }
        }
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int h = 0; h < NS; ++h) {
            s[h][0] = fast_exp2(s[h][0] - m[0]);
            s[h][1] = fast_exp2(s[h][1] - m[1]);
            s[h][2] = fast_exp2(s[h][2] - m[0]);
            s[h][3] = fast_exp2(s[h][3] - m[1]);
            ps0 += s[h][0] + s[h][2];
            ps1 += s[h][1] + s[h][3];
        }
        l[0] += ps0;
        l[1] += ps1;
        // ---- 3. P^T as the B operand: fp16, transposed 8x8 halves; 4. O^T += V^T . P^T ----
#pragma unroll
        for (int h = 0; h < NS; ++h) {
            if (NS > 1 && nv[h] == 0) continue;  // warp-uniform: nothing valid in this sub-tile
            const int rh = row0 + 16 * h;
            float w0 = 1.f, w1 = 1.f;  // INT4: each token's V scale rides on its probability
            if constexpr (KV4) {
                const float vs0 = __uint_as_float(lds32(vbase + (uint32_t)(CODE4 + (rh + r) * 4)));
                const float vs1 = __uint_as_float(lds32(vbase + (uint32_t)(CODE4 + (rh + r + 8) * 4)));
                w0 = v0[h] ? vs0 : 0.f;  // a row past the prefix may hold any scale bits
                w1 = v1[h] ? vs1 : 0.f;
            }
            const uint32_t pb0 = movmatrix_trans(pack_half2(s[h][0] * w0, s[h][1] * w0));  // tokens 2c, 2c+1
            const uint32_t pb1 = movmatrix_trans(pack_half2(s[h][2] * w1, s[h][3] * w1));  // tokens 8+2c, 8+2c+1
            const int n = nv[h];
            const bool partial = n < C::SUB;  // warp-uniform
            const uint32_t mk0 = (2 * c < n ? 0x0000ffffu : 0u) | (2 * c + 1 < n ? 0xffff0000u : 0u);
            const uint32_t mk1 = (2 * c + 8 < n ? 0x0000ffffu : 0u) | (2 * c + 9 < n ? 0xffff0000u : 0u);
            pv(vbase, rh, pb0, pb1, partial, mk0, mk1);
        }
    }

    // V^T fragment: reg 0, 1 hold tokens 2c, 2c+1; reg 2, 3 tokens 2c+8, 2c+9.
    static __device__ __forceinline__ void mask_tokens(uint32_t (&a)[4], uint32_t mk0, uint32_t mk1) {
        a[0] &= mk0;
        a[1] &= mk0;
        a[2] &= mk1;
        a[3] &= mk1;
    }

    // Output channel of O^T fragment element (m-block i, upper half h).
    __device__ __forceinline__ int out_channel(int i, int h) const {
        if (KV8 || KV4) return (D / 8) * r + 2 * i + h;
        return 16 * i + r + 8 * h;
    }

    // Write this warp's state to its slot of the merge buffer [NCW][G][D+2]:
    // (m, l, acc[D]) per row; l is summed over the 8 token rows first.
    __device__ __forceinline__ void store_state(float *merge) {
        float *mw = merge + cw * G * (D + 2);
        float ls0 = l[0], ls1 = l[1];
#pragma unroll
        for (int o_ = 4; o_ < 32; o_ <<= 1) {
            ls0 += __shfl_xor_sync(0xffffffffu, ls0, o_);
            ls1 += __shfl_xor_sync(0xffffffffu, ls1, o_);
        }
        const int q0 = 2 * c, q1 = 2 * c + 1;
        if (r == 0) {
            if (q0 < G) {
                mw[q0 * (D + 2)] = m[0];
                mw[q0 * (D + 2) + 1] = ls0;
            }
            if (q1 < G) {
                mw[q1 * (D + 2)] = m[1];
                mw[q1 * (D + 2) + 1] = ls1;
            }
        }
#pragma unroll
        for (int i = 0; i < KS; ++i) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int ch = out_channel(i, h);
                if (q0 < G) mw[q0 * (D + 2) + 2 + ch] = o[i][2 * h];
                if (q1 < G) mw[q1 * (D + 2) + 2 + ch] = o[i][2 * h + 1];
            }
        }
    }
};

}  // namespace gqaq
