// internal.h -- host-side interfaces between the C-ABI layer (abi.cu) and the
// kernel translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gqaq.h"
#include "common.cuh"

namespace gqaq {

// Encodes a 2-D fp16 tensor map: rows x cols (cols innermost), box of
// box_cols x box_rows, 128-byte swizzle or none. Returns false on failure.
bool encode_tensor_map_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                          uint32_t box_cols, uint32_t box_rows, bool swizzle128);
// K rows as a 3-D map [rows][cols/64][64], box [box_rows][cols/64][64] with
// 128-byte swizzle: one TMA load brings box_rows whole rows (all their
// 128-byte column blocks, interleaved row by row). cols: a multiple of 64.
bool encode_tensor_map_kpage(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows);
// fp32 matrix [rows][cols] (INT4 scale rows, cols * 4 a multiple of 16), box [1][box_cols].
bool encode_tensor_map_f32_rows(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols);
// Byte matrix [rows][cols] (E4M3 codes), box [box_rows][cols], swizzle 0, 64 or 128 bytes.
bool encode_tensor_map_u8(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                          int swizzle_bytes);

// Dense (page_idx == nullptr) or sparse split-context attention, one launch:
// split units are merged in-kernel by the CTA that finishes them last.
struct AttnArgs {
    const gqaq_dims *dims;
    const __half *q;
    const __half *k_cache;
    const __half *v_cache;
    const int *valid_len;
    const int *page_idx;  // sparse only
    int kpages;           // sparse only
    float scale;
    bool kv8;             // caches hold E4M3 codes
    float k_scale, v_scale;  // E4M3: value = code * scale
    bool kv4;             // caches hold INT4 levels (dense only)
    const float *k_scales, *v_scales;  // INT4: [B*Hkv][Lmax] per-token scales
    __half *out;
    void *workspace;
    size_t workspace_bytes;
};
int launch_attention(const AttnArgs &a, const LaunchCtx &ctx);
// E4M3 and INT4 cache appends (kv_lowbit.cu).
int launch_append_e4m3(const gqaq_dims *d, uint8_t *k_cache, uint8_t *v_cache, const __half *k_new,
                       const __half *v_new, const int *pos, float k_inv_scale, float v_inv_scale,
                       const LaunchCtx &ctx);
int launch_append_int4(const gqaq_dims *d, uint8_t *k_codes, float *k_scales, uint8_t *v_codes, float *v_scales,
                       const __half *k_new, const __half *v_new, const int *pos, const LaunchCtx &ctx);
// Quest over an E4M3 cache (kv_lowbit.cu): the append with the page bounds,
// the bounds rebuilt from the cache, the page scores.
int launch_append_e4m3_meta(const gqaq_dims *d, uint8_t *k_cache, uint8_t *v_cache, uint8_t *meta,
                            const __half *k_new, const __half *v_new, const int *pos, float k_inv_scale,
                            float v_inv_scale, const LaunchCtx &ctx);
int launch_update_meta_e4m3(const gqaq_dims *d, const uint8_t *k_cache, const int *valid_len, uint8_t *meta,
                            int page_begin, int page_end, const LaunchCtx &ctx);
int launch_score_pages_e4m3(const gqaq_dims *d, const __half *q, const uint8_t *meta, float k_scale,
                            const int *valid_len, float *scores, const LaunchCtx &ctx);
size_t attention_workspace_bytes(const gqaq_dims *dims, const LaunchCtx &ctx);

// Causal chunk attention (prefill.cu): q_len new tokens per sequence, the
// group axis merged into the row axis. Work items are (sequence, KV head,
// block of 128 merged rows); each is split into up to kPrefillMaxSplits
// context slices merged in-kernel. Workspace: arrival counters [items] u32
// (zero region, 256-byte rounded), then fp32 partials when split.
constexpr int kPrefillMaxSplits = 32;
struct PrefillArgs {
    const gqaq_dims *dims;
    int q_len;
    const __half *q;        // [B][Hq][q_len][D]
    const __half *k_cache;  // [B][Hkv][Lmax][D]
    const __half *v_cache;
    const int *start;       // [B]: cache row of the chunk's first token
    float scale;
    __half *out;            // [B][Hq][q_len][D]
    void *workspace;
    size_t workspace_bytes;
};
int64_t prefill_items(const gqaq_dims &dm, int q_len);
int launch_prefill(const PrefillArgs &a, const LaunchCtx &ctx);
size_t prefill_workspace_bytes(const gqaq_dims *dims, int q_len, const LaunchCtx &ctx);

// Fused Quest step (quest_fused.cu). meta == nullptr selects attention over a
// given page list (page_idx is then an input); otherwise append (pos may be
// null), score, select and attend, with scores/page_idx optional outputs.
// Workspace layout shared by the kernels that take one. A zero region comes
// first: the work ticket at kWsTicket and three words per (sequence, KV head)
// from kWsCounters (arrival counters and flags). It is zero between calls;
// every call leaves it so. Scratch follows from workspace_zero_bytes(dims).
constexpr size_t kWsTicket = 0;
constexpr size_t kWsCounters = 256;
inline size_t workspace_zero_bytes(const gqaq_dims &dm) {
    const size_t units = (size_t)dm.batch * dm.num_kv_heads;
    return (kWsCounters + 3 * units * sizeof(unsigned) + 255) & ~(size_t)255;
}

struct FusedArgs {
    const gqaq_dims *dims;
    const __half *q;
    __half *k_cache;
    __half *v_cache;
    __half *meta;
    const __half *k_new;
    const __half *v_new;
    const int *pos;
    const int *valid_len;
    int *page_idx;
    float *scores;
    int kpages;
    float scale;
    __half *out;
    void *workspace;  // work-queue kernel only
    size_t workspace_bytes;
    bool kv8;                // caches and bounds hold E4M3 codes (cluster kernel only)
    float k_inv, v_inv;      // E4M3: appended rows are quantized as fp32(x) * inv
    float k_scale, v_scale;  // E4M3: value = code value * scale
};
int launch_quest_fused(const FusedArgs &a, const LaunchCtx &ctx);
// The same step as one work queue over the whole GPU (needs the workspace).
int launch_quest_stream(const FusedArgs &a, const LaunchCtx &ctx);
// Workspace launch_quest_stream needs; 0 when the shape is outside its range.
size_t quest_stream_workspace_bytes(const gqaq_dims *dims, int kpages, const LaunchCtx &ctx);
constexpr int kFusedMaxPages = 1024;

// Quest kernels.
int launch_append_kv(const gqaq_dims *dims, __half *k_cache, __half *v_cache, __half *meta,
                     const __half *k_new, const __half *v_new, const int *pos, const LaunchCtx &ctx);
int launch_update_meta(const gqaq_dims *dims, const __half *k_cache, const int *valid_len,
                       __half *meta, int page_begin, int page_end, const LaunchCtx &ctx);
int launch_score_pages(const gqaq_dims *dims, const __half *q, const __half *meta,
                       const int *valid_len, float *scores, const LaunchCtx &ctx);
int launch_topk_pages(const gqaq_dims *dims, const float *scores, const int *valid_len, int k,
                      int *page_idx, const LaunchCtx &ctx);

// Largest Pmax the top-K kernel keeps in shared memory.
constexpr int kTopkMaxPages = 32768;

}  // namespace gqaq
