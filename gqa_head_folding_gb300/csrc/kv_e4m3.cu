// kv_e4m3.cu -- append to an E4M3 (8-bit floating point) KV cache.
//
// The Quest review names the cache update path and lower-precision (fp8 /
// 4-bit) KV caches as the next steps. This file holds the 8-bit cache's
// append: the new token's k and v rows, fp16, become E4M3 codes
// RNE-satfinite(fp32(x) * inv_scale) at row pos[b] of every KV head. The
// attention over such a cache is attn_partial_kernel<D, G, false, true>.
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

}  // namespace

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
