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
// The attention over either cache is attn_partial_kernel<D, G, false, KV>.
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

}  // namespace gqaq
