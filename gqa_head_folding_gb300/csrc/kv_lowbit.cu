// kv_lowbit.cu -- appends to the 8-bit (E4M3) and 4-bit (INT4) KV caches.
//
// Neither source page defines a low-bit KV cache. The OPT post's section 5
// ("KV Cache Update Operations Remain") names the cache-write path as the
// next target; the Quest review states that its 4-bit figure is weight
// quantization, not KV storage. The two formats here are this library's own
// plainest choices. Each append turns the new token's fp16
// k and v rows into the cache format at row pos[b] of every KV head:
//  - E4M3: codes RNE-satfinite(fp32(x) * inv_scale), one scale per tensor;
//  - INT4: per row scale = amax / 7, levels clamp(rne(x / scale), -7, 7)
//    stored as nibbles level + 8, the scale beside the row.
// The attention over either cache is attn_partial_kernel<D, G, false, KV>;
// over the selected pages of an E4M3 cache, attn_partial_kernel<D, G, true, 1>.
// The Quest page bounds and scores of an E4M3 cache are below as well.
#include "internal.h"

namespace gqaq {
namespace {

struct Append8Params {
    uint8_t *k_cache, *v_cache;
    const __half *k_new, *v_new;
    const int *pos;
    int *status;
    int B, Hkv, Lmax, D;
    float k_inv, v_inv;
};

// Two fp32 values -> E4M3 codes, `lo` in the low byte: round to nearest
// even, magnitudes beyond 448 saturated.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(r)
        : "f"(lo), "f"(hi));
    return r;
}

// One CTA per (sequence, KV head); each thread quantizes channel pairs.
__global__ void __launch_bounds__(64) append_e4m3_kernel(const Append8Params p) {
    pdl_wait_and_release();
    const int unit = blockIdx.x;
    const int b = unit / p.Hkv, kv = unit - (unit / p.Hkv) * p.Hkv;
    const int pos = p.pos[b];
    if (pos < 0 || pos >= p.Lmax) {
        if (threadIdx.x == 0 && kv == 0) raise_flag(p.status, GQAQ_DEV_BAD_POS);
        return;
    }
    const int64_t row = ((int64_t)unit * p.Lmax + pos) * p.D;
    const __half2 *kn = reinterpret_cast<const __half2 *>(p.k_new + (int64_t)unit * p.D);
    const __half2 *vn = reinterpret_cast<const __half2 *>(p.v_new + (int64_t)unit * p.D);
    for (int c = threadIdx.x; c < p.D / 2; c += blockDim.x) {
        const float2 k = __half22float2(kn[c]);
        const float2 v = __half22float2(vn[c]);
        reinterpret_cast<uint16_t *>(p.k_cache + row)[c] = (uint16_t)f32x2_to_e4m3x2(k.x * p.k_inv, k.y * p.k_inv);
        reinterpret_cast<uint16_t *>(p.v_cache + row)[c] = (uint16_t)f32x2_to_e4m3x2(v.x * p.v_inv, v.y * p.v_inv);
    }
}

struct Append4Params {
    uint8_t *k_codes, *v_codes;
    float *k_scales, *v_scales;
    const __half *k_new, *v_new;
    const int *pos;
    int *status;
    int B, Hkv, Lmax;
};

// One row of D channels -> (D/2 code bytes, scale), by one warp. CPL = D/32
// channels per lane (2 or 4, consecutive); IEEE divisions, ties to even.
template <int D>
__device__ __forceinline__ void quantize_row4(const __half *x, uint8_t *codes, float *scale, int lane) {
    constexpr int CPL = D / 32;
    float v[CPL];
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < CPL; ++e) {
        v[e] = __half2float(x[lane * CPL + e]);
        amax = fmaxf(amax, fabsf(v[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = __fdiv_rn(amax, 7.0f);
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < CPL; ++e) {
        int q = 0;
        if (sc > 0.f) {
            const float t = rintf(__fdiv_rn(v[e], sc));
            q = t > 7.f ? 7 : (t < -7.f ? -7 : (int)t);
        }
        packed |= (uint32_t)(q + 8) << (4 * e);
    }
    if (CPL == 2) codes[lane] = (uint8_t)packed;
    else reinterpret_cast<uint16_t *>(codes)[lane] = (uint16_t)packed;
    if (lane == 0) *scale = sc;
}

// One warp per (sequence, KV head): the K row, then the V row.
template <int D>
__global__ void __launch_bounds__(128) append_int4_kernel(const Append4Params p) {
    pdl_wait_and_release();
    const int unit = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (unit >= p.B * p.Hkv) return;
    const int b = unit / p.Hkv;
    const int pos = p.pos[b];
    if (pos < 0 || pos >= p.Lmax) {
        if (lane == 0 && unit % p.Hkv == 0) raise_flag(p.status, GQAQ_DEV_BAD_POS);
        return;
    }
    const int64_t row = (int64_t)unit * p.Lmax + pos;
    quantize_row4<D>(p.k_new + (int64_t)unit * D, p.k_codes + row * (D / 2), p.k_scales + row, lane);
    quantize_row4<D>(p.v_new + (int64_t)unit * D, p.v_codes + row * (D / 2), p.v_scales + row, lane);
}

// ---------------------------------------------------------------------------
// Quest over an E4M3 cache ("Quest ..." review, page-score section): page
// min/max kept as E4M3 codes of the keys' values (compared after decoding; a
// zero bound is stored as the code 0x00, so each bound has one code), and the
// page score U = sum_i max(q_i m_i, q_i M_i) on the code values, times the
// positive K scale (the ranking is the same as on the dequantized keys).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 e4m3x2_value(uint32_t two) {
    uint32_t h;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(two));
    return __half22float2(*reinterpret_cast<__half2 *>(&h));
}
__device__ __forceinline__ float e4m3_value(uint32_t code) { return e4m3x2_value(code & 0xffu).x; }
__device__ __forceinline__ uint32_t canonical_e4m3(uint32_t code) { return (code & 0x7fu) == 0u ? 0u : code; }

struct Append8MetaParams {
    uint8_t *k_cache, *v_cache, *meta;
    const __half *k_new, *v_new;
    const int *pos;
    int *status;
    int B, Hkv, Lmax, Pmax, S;
    float k_inv, v_inv;
};

// One warp per (sequence, KV head); lane l owns channels [l*CPL, (l+1)*CPL).
// The codes are those of append_e4m3_kernel; then the page's bounds.
template <int D>
__global__ void __launch_bounds__(128) append_e4m3_meta_kernel(const Append8MetaParams p) {
    pdl_wait_and_release();
    constexpr int CPL = D / 32;  // 2 or 4
    const int u = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (u >= p.B * p.Hkv) return;
    const int b = u / p.Hkv;
    const int pos = p.pos[b];
    if (pos < 0 || pos >= p.Lmax) {
        if (lane == 0 && (u % p.Hkv) == 0) raise_flag(p.status, GQAQ_DEV_BAD_POS);
        return;
    }
    const int c0 = lane * CPL;
    uint32_t kc = 0, vc = 0;  // CPL codes, channel c0 in the low byte
#pragma unroll
    for (int e = 0; e < CPL; e += 2) {
        const float2 k = __half22float2(*reinterpret_cast<const __half2 *>(p.k_new + (int64_t)u * D + c0 + e));
        const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(p.v_new + (int64_t)u * D + c0 + e));
        kc |= f32x2_to_e4m3x2(k.x * p.k_inv, k.y * p.k_inv) << (8 * e);
        vc |= f32x2_to_e4m3x2(v.x * p.v_inv, v.y * p.v_inv) << (8 * e);
    }
    const int64_t row = ((int64_t)u * p.Lmax + pos) * D + c0;
    if (CPL == 4) {
        *reinterpret_cast<uint32_t *>(p.k_cache + row) = kc;
        *reinterpret_cast<uint32_t *>(p.v_cache + row) = vc;
    } else {
        *reinterpret_cast<uint16_t *>(p.k_cache + row) = (uint16_t)kc;
        *reinterpret_cast<uint16_t *>(p.v_cache + row) = (uint16_t)vc;
    }
    uint8_t *mrow = p.meta + ((int64_t)u * p.Pmax + pos / p.S) * 2 * D;
    const bool fresh = (pos % p.S) == 0;
#pragma unroll
    for (int e = 0; e < CPL; ++e) {
        const uint32_t c = (kc >> (8 * e)) & 0xffu;
        uint32_t mn = canonical_e4m3(c), mx = mn;
        if (!fresh) {
            const uint32_t om = mrow[c0 + e], oM = mrow[D + c0 + e];
            const float x = e4m3_value(c);
            mn = x < e4m3_value(om) ? mn : om;
            mx = x > e4m3_value(oM) ? mx : oM;
        }
        mrow[c0 + e] = (uint8_t)mn;
        mrow[D + c0 + e] = (uint8_t)mx;
    }
}

struct Meta8Params {
    const uint8_t *k_cache;
    const int *valid_len;
    uint8_t *meta;
    int *status;
    int B, Hkv, Lmax, Pmax, S, p0, p1;
};

// Page bounds from the cache for pages [p0, p1). One warp per page.
template <int D>
__global__ void __launch_bounds__(256) update_meta_e4m3_kernel(const Meta8Params p) {
    pdl_wait_and_release();
    constexpr int CPL = D / 32;
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
    const uint8_t *kr = p.k_cache + (u * p.Lmax) * D + lane * CPL;
    uint32_t cmn[CPL], cmx[CPL];
    float vmn[CPL], vmx[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) {
        cmn[e] = cmx[e] = kr[(int64_t)t0 * D + e];
        vmn[e] = vmx[e] = e4m3_value(cmn[e]);
    }
    for (int t = t0 + 1; t < t1; ++t) {
#pragma unroll
        for (int e = 0; e < CPL; ++e) {
            const uint32_t c = kr[(int64_t)t * D + e];
            const float x = e4m3_value(c);
            if (x < vmn[e]) { vmn[e] = x; cmn[e] = c; }
            if (x > vmx[e]) { vmx[e] = x; cmx[e] = c; }
        }
    }
    uint8_t *mrow = p.meta + (u * p.Pmax + page) * 2 * D + lane * CPL;
#pragma unroll
    for (int e = 0; e < CPL; ++e) {
        mrow[e] = (uint8_t)canonical_e4m3(cmn[e]);
        mrow[D + e] = (uint8_t)canonical_e4m3(cmx[e]);
    }
}

struct Score8Params {
    const __half *q;
    const uint8_t *meta;
    const int *valid_len;
    float *scores;
    int *status;
    int B, Hkv, Lmax, Pmax, S;
    float k_scale;
};

// Page scores over E4M3 bounds. CTA (x, unit) scores pages [64x, 64x + 64):
// warp w pages 8w..8w+7, LPP lanes per page record of 2D bytes ([m codes; M
// codes]), each lane one 16-byte chunk against the matching channels of
// [min(q,0); max(q,0)] (staged in fp32), reduced over the LPP lanes; the
// largest U over the G query rows, times the K scale.
template <int D, int G>
__global__ void __launch_bounds__(256) score_e4m3_kernel(const Score8Params p) {
    constexpr int LPP = 2 * D / 16;  // 16 (D = 128) or 8 (D = 64)
    constexpr int PPI = 32 / LPP;    // pages a warp scores at once
    constexpr int NIT = 8 / PPI;     // rounds per warp
    __shared__ __align__(16) float qs[G][2 * D];
    pdl_wait_and_release();
    const int u = blockIdx.y;
    const int b = u / p.Hkv, kv = u - (u / p.Hkv) * p.Hkv;
    const int raw = p.valid_len[b];
    if (threadIdx.x == 0 && blockIdx.x == 0 && kv == 0 && (raw < 1 || raw > p.Lmax))
        raise_flag(p.status, GQAQ_DEV_BAD_LEN);
    const int P = (clamp_len(raw, p.Lmax) + p.S - 1) / p.S;
    const int pg0 = blockIdx.x * 64;
    if (pg0 >= P) return;
    const __half *qg = p.q + ((int64_t)b * p.Hkv * G + (int64_t)kv * G) * D;
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
        const int g = i / D, c = i - (i / D) * D;
        const float x = __half2float(qg[(int64_t)g * D + c]);
        qs[g][c] = fminf(x, 0.f);
        qs[g][D + c] = fmaxf(x, 0.f);
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / LPP, j = lane - (lane / LPP) * LPP;
    uint4 w[NIT];
#pragma unroll
    for (int it = 0; it < NIT; ++it) {  // every load first, then the arithmetic
        const int page = pg0 + warp * 8 + it * PPI + sub;
        w[it] = page < P ? *reinterpret_cast<const uint4 *>(p.meta + ((int64_t)u * p.Pmax + page) * 2 * D + 16 * j)
                         : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int page = pg0 + warp * 8 + it * PPI + sub;
        float v[16];
        const uint32_t wd[4] = {w[it].x, w[it].y, w[it].z, w[it].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 lo = e4m3x2_value(wd[k] & 0xffffu), hi = e4m3x2_value(wd[k] >> 16);
            v[4 * k] = lo.x;
            v[4 * k + 1] = lo.y;
            v[4 * k + 2] = hi.x;
            v[4 * k + 3] = hi.y;
        }
        float best = -INFINITY;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float4 *qv = reinterpret_cast<const float4 *>(&qs[g][16 * j]);
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 qq = qv[k];
                acc = fmaf(qq.x, v[4 * k], acc);
                acc = fmaf(qq.y, v[4 * k + 1], acc);
                acc = fmaf(qq.z, v[4 * k + 2], acc);
                acc = fmaf(qq.w, v[4 * k + 3], acc);
            }
#pragma unroll
            for (int o = LPP / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            best = fmaxf(best, acc);
        }
        if (j == 0 && page < P) p.scores[(int64_t)u * p.Pmax + page] = best * p.k_scale;
    }
}

}  // namespace

int launch_append_int4(const gqaq_dims *d, uint8_t *k_codes, float *k_scales, uint8_t *v_codes, float *v_scales,
                       const __half *k_new, const __half *v_new, const int *pos, const LaunchCtx &ctx) {
    Append4Params p;
    p.k_codes = k_codes;
    p.v_codes = v_codes;
    p.k_scales = k_scales;
    p.v_scales = v_scales;
    p.k_new = k_new;
    p.v_new = v_new;
    p.pos = pos;
    p.status = ctx.status;
    p.B = d->batch;
    p.Hkv = d->num_kv_heads;
    p.Lmax = d->max_len;
    const dim3 grid((unsigned)((d->batch * d->num_kv_heads + 3) / 4));
    cudaError_t e;
    if (d->head_dim == 64) e = launch_kernel(append_int4_kernel<64>, grid, dim3(128), 0, ctx, 0, p);
    else if (d->head_dim == 128) e = launch_kernel(append_int4_kernel<128>, grid, dim3(128), 0, ctx, 0, p);
    else return GQAQ_ERR_UNSUPPORTED;
    return e == cudaSuccess ? GQAQ_OK : GQAQ_ERR_CUDA;
}

int launch_append_e4m3(const gqaq_dims *d, uint8_t *k_cache, uint8_t *v_cache, const __half *k_new,
                       const __half *v_new, const int *pos, float k_inv_scale, float v_inv_scale,
                       const LaunchCtx &ctx) {
    Append8Params p;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.k_new = k_new;
    p.v_new = v_new;
    p.pos = pos;
    p.status = ctx.status;
    p.B = d->batch;
    p.Hkv = d->num_kv_heads;
    p.Lmax = d->max_len;
    p.D = d->head_dim;
    p.k_inv = k_inv_scale;
    p.v_inv = v_inv_scale;
    if (launch_kernel(append_e4m3_kernel, dim3(d->batch * d->num_kv_heads), dim3(64), 0, ctx, 0, p) != cudaSuccess)
        return GQAQ_ERR_CUDA;
    return GQAQ_OK;
}

int launch_append_e4m3_meta(const gqaq_dims *d, uint8_t *k_cache, uint8_t *v_cache, uint8_t *meta,
                            const __half *k_new, const __half *v_new, const int *pos, float k_inv_scale,
                            float v_inv_scale, const LaunchCtx &ctx) {
    Append8MetaParams p;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.meta = meta;
    p.k_new = k_new;
    p.v_new = v_new;
    p.pos = pos;
    p.status = ctx.status;
    p.B = d->batch;
    p.Hkv = d->num_kv_heads;
    p.Lmax = d->max_len;
    p.S = d->page_size;
    p.Pmax = (d->max_len + d->page_size - 1) / d->page_size;
    p.k_inv = k_inv_scale;
    p.v_inv = v_inv_scale;
    const int units = d->batch * d->num_kv_heads;
    const dim3 grid((units + 3) / 4);
    cudaError_t e = d->head_dim == 128 ? launch_kernel(append_e4m3_meta_kernel<128>, grid, dim3(128), 0, ctx, 0, p)
                                       : launch_kernel(append_e4m3_meta_kernel<64>, grid, dim3(128), 0, ctx, 0, p);
    return e == cudaSuccess ? GQAQ_OK : GQAQ_ERR_CUDA;
}

int launch_update_meta_e4m3(const gqaq_dims *d, const uint8_t *k_cache, const int *valid_len, uint8_t *meta,
                            int page_begin, int page_end, const LaunchCtx &ctx) {
    if (page_end <= page_begin) return GQAQ_OK;
    Meta8Params p;
    p.k_cache = k_cache;
    p.valid_len = valid_len;
    p.meta = meta;
    p.status = ctx.status;
    p.B = d->batch;
    p.Hkv = d->num_kv_heads;
    p.Lmax = d->max_len;
    p.S = d->page_size;
    p.Pmax = (d->max_len + d->page_size - 1) / d->page_size;
    p.p0 = page_begin;
    p.p1 = page_end;
    const int64_t warps = (int64_t)d->batch * d->num_kv_heads * (page_end - page_begin);
    const dim3 grid((unsigned)((warps + 7) / 8));
    cudaError_t e = d->head_dim == 128 ? launch_kernel(update_meta_e4m3_kernel<128>, grid, dim3(256), 0, ctx, 0, p)
                                       : launch_kernel(update_meta_e4m3_kernel<64>, grid, dim3(256), 0, ctx, 0, p);
    return e == cudaSuccess ? GQAQ_OK : GQAQ_ERR_CUDA;
}

namespace {
template <int D>
cudaError_t score8_g(const Score8Params &p, int G, dim3 grid, const LaunchCtx &ctx) {
    switch (G) {
        case 1: return launch_kernel(score_e4m3_kernel<D, 1>, grid, dim3(256), 0, ctx, 0, p);
        case 2: return launch_kernel(score_e4m3_kernel<D, 2>, grid, dim3(256), 0, ctx, 0, p);
        case 4: return launch_kernel(score_e4m3_kernel<D, 4>, grid, dim3(256), 0, ctx, 0, p);
        default: return launch_kernel(score_e4m3_kernel<D, 8>, grid, dim3(256), 0, ctx, 0, p);
    }
}
}  // namespace

int launch_score_pages_e4m3(const gqaq_dims *d, const __half *q, const uint8_t *meta, float k_scale,
                            const int *valid_len, float *scores, const LaunchCtx &ctx) {
    Score8Params p;
    p.q = q;
    p.meta = meta;
    p.valid_len = valid_len;
    p.scores = scores;
    p.status = ctx.status;
    p.B = d->batch;
    p.Hkv = d->num_kv_heads;
    p.Lmax = d->max_len;
    p.S = d->page_size;
    p.Pmax = (d->max_len + d->page_size - 1) / d->page_size;
    p.k_scale = k_scale;
    const int G = d->num_q_heads / d->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return GQAQ_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)((p.Pmax + 63) / 64), (unsigned)(d->batch * d->num_kv_heads));
    const cudaError_t e = d->head_dim == 128 ? score8_g<128>(p, G, grid, ctx) : score8_g<64>(p, G, grid, ctx);
    return e == cudaSuccess ? GQAQ_OK : GQAQ_ERR_CUDA;
}

}  // namespace gqaq
