// quest_tile.cuh -- page scoring from a metadata tile in shared memory,
// shared by the Quest kernels.
//
// "Quest: Query-Aware Sparsity ..." (review), page-score section:
//   U(p, q) = sum_i max(q_i * m_{p,i}, q_i * M_{p,i}).
// Since m_{p,i} <= M_{p,i}, the larger product takes M where q_i > 0 and m
// where q_i < 0, so U = [min(q, 0); max(q, 0)] . [m; M], a dot product of
// length 2D. With grouped query heads ("Core ML Decode Optimization ...",
// section 3) a KV head's page score is the largest U over its G query rows.
#pragma once

#include "common.cuh"

namespace gqaq {

// fp32 score -> u32 key whose unsigned order is the float order (-0 == +0).
__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t x = __float_as_uint(f);
    if (x == 0x80000000u) x = 0u;  // -0 ranks with +0
    return (x & 0x80000000u) ? ~x : (x | 0x80000000u);
}
__device__ __forceinline__ uint32_t hmin0_bits(uint32_t x) {
    __half2 h = *reinterpret_cast<__half2 *>(&x);
    __half2 r = __hmin2(h, __float2half2_rn(0.f));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t hmax0_bits(uint32_t x) {
    __half2 h = *reinterpret_cast<__half2 *>(&x);
    __half2 r = __hmax2(h, __float2half2_rn(0.f));
    return *reinterpret_cast<uint32_t *>(&r);
}

// One consumer warp scores 8 pages per pass of a metadata tile. The tile
// holds MT page records [m (D halves) | M (D halves)] as 2D/64 column blocks
// of MT rows x 128 bytes, 128-byte swizzled (TMA SWIZZLE_128B). Lane =
// 8 * quarter + page: quarters 0-1 dot min(q,0) with the two halves of m,
// quarters 2-3 dot max(q,0) with the two halves of M.
template <int D, int G, int MT>
struct MetaScorer {
    static constexpr int MBLK = MT * 128;
    static constexpr int NCHQ = D / 16;          // 16-byte chunks per record quarter
    static constexpr bool QTREG = (G * D <= 512);
    static constexpr int GQT = QTREG ? G : 4;    // query rows per register pass
    static constexpr int NPASST = G / GQT;
    static constexpr int QT_BYTES = G * 2 * D * 2;  // [G][2D] fp16 [q_neg | q_pos] when not in registers

    int jp, qq, cq0, qch0;
    bool negq;
    uint4 qt[GQT][NCHQ];

    __device__ __forceinline__ void init(int lane) {
        jp = lane & 7;
        qq = lane >> 3;
        cq0 = qq * (D / 2);
        negq = qq < 2;
        qch0 = (qq & 1) * (D / 2);
    }
    // Registers (QTREG): this lane's quarter of [q_neg | q_pos] for all G rows.
    __device__ __forceinline__ void load_q_regs(const __half *qg) {
#pragma unroll
        for (int g = 0; g < GQT; ++g)
#pragma unroll
            for (int c = 0; c < NCHQ; ++c) {
                const uint4 v = *reinterpret_cast<const uint4 *>(qg + g * D + qch0 + c * 8);
                qt[g][c] = negq ? make_uint4(hmin0_bits(v.x), hmin0_bits(v.y), hmin0_bits(v.z), hmin0_bits(v.w))
                                : make_uint4(hmax0_bits(v.x), hmax0_bits(v.y), hmax0_bits(v.z), hmax0_bits(v.w));
            }
    }
    // Shared memory (not QTREG): threads tid of nthreads fill [G][2D].
    __device__ __forceinline__ static void load_q_smem(const __half *qg, __half *qt_s, int tid, int nthreads) {
        for (int e = tid; e < G * D / 8; e += nthreads) {
            const int g = e / (D / 8), c = e % (D / 8);
            const uint4 v = *reinterpret_cast<const uint4 *>(qg + g * D + c * 8);
            reinterpret_cast<uint4 *>(qt_s + g * 2 * D)[c] =
                make_uint4(hmin0_bits(v.x), hmin0_bits(v.y), hmin0_bits(v.z), hmin0_bits(v.w));
            reinterpret_cast<uint4 *>(qt_s + g * 2 * D + D)[c] =
                make_uint4(hmax0_bits(v.x), hmax0_bits(v.y), hmax0_bits(v.z), hmax0_bits(v.w));
        }
    }
    // Score of tile row `row` (page jp of this pass), max over the G rows; the
    // value is complete in every lane of the page's four quarters.
    __device__ __forceinline__ float score(uint32_t sbase, int row, const __half *qt_s) {
        const uint32_t base = sbase + (uint32_t)((cq0 / 64) * MBLK + row * 128);
        const uint32_t x0 = (uint32_t)(((cq0 % 64) / 8) ^ (row & 7));
        float uu[G];
#pragma unroll
        for (int ps = 0; ps < NPASST; ++ps) {
            if (!QTREG) {
#pragma unroll
                for (int g = 0; g < GQT; ++g)
#pragma unroll
                    for (int c = 0; c < NCHQ; ++c)
                        qt[g][c] = lds128(smem_u32(qt_s + (ps * GQT + g) * 2 * D + cq0 + c * 8));
            }
            float a0[GQT], a1[GQT];
#pragma unroll
            for (int g = 0; g < GQT; ++g) a0[g] = a1[g] = 0.f;
#pragma unroll
            for (int c = 0; c < NCHQ; ++c) {
                const uint4 mc = lds128(base + ((x0 ^ (uint32_t)c) << 4));
#pragma unroll
                for (int g = 0; g < GQT; ++g) {
                    a0[g] = fma_h_lo(qt[g][c].x, mc.x, a0[g]);
                    a1[g] = fma_h_hi(qt[g][c].x, mc.x, a1[g]);
                    a0[g] = fma_h_lo(qt[g][c].y, mc.y, a0[g]);
                    a1[g] = fma_h_hi(qt[g][c].y, mc.y, a1[g]);
                    a0[g] = fma_h_lo(qt[g][c].z, mc.z, a0[g]);
                    a1[g] = fma_h_hi(qt[g][c].z, mc.z, a1[g]);
                    a0[g] = fma_h_lo(qt[g][c].w, mc.w, a0[g]);
                    a1[g] = fma_h_hi(qt[g][c].w, mc.w, a1[g]);
                }
            }
#pragma unroll
            for (int g = 0; g < GQT; ++g) uu[ps * GQT + g] = a0[g] + a1[g];
        }
        float best = -INFINITY;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float x = uu[g];
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            best = fmaxf(best, x);
        }
        return best;
    }
    // Same score with [q_neg | q_pos] ([G][2D] fp16) read from shared memory
    // chunk by chunk, so no query registers stay live between calls.
    __device__ __forceinline__ float score_qs(uint32_t sbase, int row, const __half *qt_s) {
        const uint32_t base = sbase + (uint32_t)((cq0 / 64) * MBLK + row * 128);
        const uint32_t x0 = (uint32_t)(((cq0 % 64) / 8) ^ (row & 7));
        const uint32_t qbase = smem_u32(qt_s + cq0);
        float a0[G], a1[G];
#pragma unroll
        for (int g = 0; g < G; ++g) a0[g] = a1[g] = 0.f;
#pragma unroll
        for (int c = 0; c < NCHQ; ++c) {
            const uint4 mc = lds128(base + ((x0 ^ (uint32_t)c) << 4));
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint4 qv = lds128(qbase + (uint32_t)((g * 2 * D + c * 8) * 2));
                a0[g] = fma_h_lo(qv.x, mc.x, a0[g]);
                a1[g] = fma_h_hi(qv.x, mc.x, a1[g]);
                a0[g] = fma_h_lo(qv.y, mc.y, a0[g]);
                a1[g] = fma_h_hi(qv.y, mc.y, a1[g]);
                a0[g] = fma_h_lo(qv.z, mc.z, a0[g]);
                a1[g] = fma_h_hi(qv.z, mc.z, a1[g]);
                a0[g] = fma_h_lo(qv.w, mc.w, a0[g]);
                a1[g] = fma_h_hi(qv.w, mc.w, a1[g]);
            }
        }
        float best = -INFINITY;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float x = a0[g] + a1[g];
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            best = fmaxf(best, x);
        }
        return best;
    }
};

}  // namespace gqaq
