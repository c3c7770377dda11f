// abi.cu -- the extern "C" entry points declared in include/gqaq.h: host-side
// argument validation, per-device launch context, TMA descriptor encoding,
// options and the device status word.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "internal.h"

namespace gqaq {

// Device status word, one per device that loads the library.
__device__ int g_device_status = 0;

namespace {

constexpr int kMaxDevices = 64;

std::atomic<int64_t> g_opt_max_ctas{0};
std::atomic<int64_t> g_opt_timeout_ns{2000000000LL};
std::atomic<int64_t> g_opt_test_stall{0};
std::atomic<int64_t> g_opt_cluster_size{0};
std::atomic<int64_t> g_opt_pdl{1};
std::atomic<int64_t> g_opt_quest_early_meta{0};
std::atomic<int64_t> g_opt_dense_early_kv{0};
std::atomic<int64_t> g_opt_quest_kernel{0};
std::atomic<int64_t> g_opt_prefill_splits{0};
std::atomic<int64_t> g_opt_prefill_kernel{0};

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    int *status = nullptr;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mutex;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// Per-device set-up: SM count and the device address of the status word.
int device_state(DeviceState **out, int *dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GQAQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GQAQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceState &s = g_dev[dev];
    if (!s.ready) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GQAQ_ERR_CUDA;
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess || addr == nullptr)
            return GQAQ_ERR_CUDA;
        s.num_sms = sms;
        s.status = static_cast<int *>(addr);
        s.ready = true;
    }
    *out = &s;
    *dev_out = dev;
    return GQAQ_OK;
}

int make_ctx(LaunchCtx *ctx, void *stream) {
    DeviceState *s = nullptr;
    int dev = 0;
    const int rc = device_state(&s, &dev);
    if (rc != GQAQ_OK) return rc;
    ctx->stream = static_cast<cudaStream_t>(stream);
    ctx->device = dev;
    ctx->num_sms = s->num_sms;
    ctx->max_ctas = (int)g_opt_max_ctas.load();
    ctx->timeout_ns = (uint64_t)g_opt_timeout_ns.load();
    ctx->test_stall = (int)g_opt_test_stall.load();
    ctx->cluster_size = (int)g_opt_cluster_size.load();
    ctx->pdl = (int)g_opt_pdl.load();
    ctx->quest_kernel = (int)g_opt_quest_kernel.load();
    ctx->prefill_splits = (int)g_opt_prefill_splits.load();
    ctx->prefill_kernel = (int)g_opt_prefill_kernel.load();
    ctx->quest_early_meta = (int)g_opt_quest_early_meta.load();
    ctx->dense_early_kv = (int)g_opt_dense_early_kv.load();
    ctx->status = s->status;
    return GQAQ_OK;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by every entry point.
int check_dims(const gqaq_dims *d, bool quest) {
    if (d == nullptr) return GQAQ_ERR_INVALID_ARG;
    if (d->batch < 1 || d->num_q_heads < 1 || d->num_kv_heads < 1 || d->max_len < 1 || d->head_dim < 1)
        return GQAQ_ERR_INVALID_ARG;
    if (d->num_q_heads % d->num_kv_heads != 0) return GQAQ_ERR_INVALID_ARG;
    if (quest && d->page_size < 1) return GQAQ_ERR_INVALID_ARG;
    const int G = d->num_q_heads / d->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return GQAQ_ERR_UNSUPPORTED;
    if (d->head_dim != 64 && d->head_dim != 128) return GQAQ_ERR_UNSUPPORTED;
    if (quest && d->page_size != 8 && d->page_size != 16 && d->page_size != 32 && d->page_size != 64)
        return GQAQ_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)d->batch * d->num_kv_heads * d->max_len;
    if (rows > (int64_t)INT32_MAX - 1024) return GQAQ_ERR_UNSUPPORTED;
    return GQAQ_OK;
}

}  // namespace

bool encode_tensor_map_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                          uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (g_encode == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides,
                                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_tensor_map_u8(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                          int swizzle_bytes) {
    if (!encode_tensor_map_2d(map, base, rows, cols, cols, box_rows, false)) return false;  // loads g_encode
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {(cuuint32_t)cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                        : CU_TENSOR_MAP_SWIZZLE_NONE;
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_tensor_map_f32_rows(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols) {
    if ((cols * 4) % 16 != 0) return false;
    if (!encode_tensor_map_2d(map, base, rows, cols * 2, 64, 1, false)) return false;  // loads g_encode
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 4};
    const cuuint32_t box[2] = {box_cols, 1};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_tensor_map_kpage(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    if (cols % 64 != 0 || !encode_tensor_map_2d(map, base, rows, cols, 64, box_rows, true)) return false;  // loads g_encode
    const cuuint64_t dims[3] = {64, cols / 64, rows};
    const cuuint64_t strides[2] = {128, cols * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)(cols / 64), box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace gqaq

using namespace gqaq;

extern "C" {

int gqaq_version(void) { return 100; }

const char *gqaq_status_string(int status) {
    switch (status) {
        case GQAQ_OK: return "GQAQ_OK";
        case GQAQ_ERR_INVALID_ARG: return "GQAQ_ERR_INVALID_ARG";
        case GQAQ_ERR_UNSUPPORTED: return "GQAQ_ERR_UNSUPPORTED";
        case GQAQ_ERR_WORKSPACE: return "GQAQ_ERR_WORKSPACE";
        case GQAQ_ERR_CUDA: return "GQAQ_ERR_CUDA";
        case GQAQ_ERR_TIMEOUT: return "GQAQ_ERR_TIMEOUT";
        default: return "GQAQ_ERR_UNKNOWN";
    }
}

int gqaq_set_option(int option, int64_t value) {
    switch (option) {
        case GQAQ_OPT_MAX_CTAS:
            if (value < 0 || value > INT32_MAX) return GQAQ_ERR_INVALID_ARG;
            g_opt_max_ctas.store(value);
            return GQAQ_OK;
        case GQAQ_OPT_WAIT_TIMEOUT_NS:
            if (value < 0) return GQAQ_ERR_INVALID_ARG;
            g_opt_timeout_ns.store(value);
            return GQAQ_OK;
        case GQAQ_OPT_TEST_STALL:
            g_opt_test_stall.store(value != 0 ? 1 : 0);
            return GQAQ_OK;
        case GQAQ_OPT_PDL:
            g_opt_pdl.store(value != 0 ? 1 : 0);
            return GQAQ_OK;
        case GQAQ_OPT_QUEST_KERNEL:
            if (value < 0 || value > 2) return GQAQ_ERR_INVALID_ARG;
            g_opt_quest_kernel.store(value);
            return GQAQ_OK;
        case GQAQ_OPT_PREFILL_SPLITS:
            if (value < 0 || value > kPrefillMaxSplits) return GQAQ_ERR_INVALID_ARG;
            g_opt_prefill_splits.store(value);
            return GQAQ_OK;
        case GQAQ_OPT_PREFILL_KERNEL:
            if (value < 0 || value > 2) return GQAQ_ERR_INVALID_ARG;
            g_opt_prefill_kernel.store(value);
            return GQAQ_OK;
        case GQAQ_OPT_DENSE_EARLY_KV:
            if (value != 0 && value != 1) return GQAQ_ERR_INVALID_ARG;
            g_opt_dense_early_kv.store(value);
            return GQAQ_OK;
        case GQAQ_OPT_QUEST_EARLY_META:
            if (value != 0 && value != 1) return GQAQ_ERR_INVALID_ARG;
            g_opt_quest_early_meta.store(value);
            return GQAQ_OK;
        case GQAQ_OPT_CLUSTER_SIZE:
            if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8) return GQAQ_ERR_INVALID_ARG;
            g_opt_cluster_size.store(value);
            return GQAQ_OK;
        default:
            return GQAQ_ERR_INVALID_ARG;
    }
}

int gqaq_device_status(int *flags, int reset) {
    if (flags == nullptr) return GQAQ_ERR_INVALID_ARG;
    LaunchCtx ctx;
    const int rc = make_ctx(&ctx, nullptr);
    if (rc != GQAQ_OK) return rc;
    if (cudaDeviceSynchronize() != cudaSuccess) return GQAQ_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, ctx.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GQAQ_ERR_CUDA;
    if (reset) {
        const int zero = 0;
        if (cudaMemcpy(ctx.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return GQAQ_ERR_CUDA;
    }
    *flags = v;
    return (v & GQAQ_DEV_TIMEOUT) ? GQAQ_ERR_TIMEOUT : GQAQ_OK;
}

size_t gqaq_workspace_bytes(const gqaq_dims *dims, int max_selected_pages) {
    if (check_dims(dims, false) != GQAQ_OK) return 0;
    LaunchCtx ctx;
    if (make_ctx(&ctx, nullptr) != GQAQ_OK) return 0;
    size_t need = attention_workspace_bytes(dims, ctx);
    if (need == 0) return 0;
    if (max_selected_pages > 0 && check_dims(dims, true) == GQAQ_OK) {
        const size_t qs = quest_stream_workspace_bytes(dims, max_selected_pages, ctx);
        if (qs > need) need = qs;
    }
    return need;
}

int gqa_decode_attn(const gqaq_dims *dims, const gqaq_half *q, const gqaq_half *k_cache,
                    const gqaq_half *v_cache, const int32_t *valid_len, float scale, gqaq_half *out,
                    void *workspace, size_t workspace_bytes, void *stream) {
    int rc = check_dims(dims, false);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        !aligned16(valid_len))
        return GQAQ_ERR_INVALID_ARG;
    if (!isfinite(scale)) return GQAQ_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned16(workspace)) return GQAQ_ERR_WORKSPACE;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    AttnArgs a = {};
    a.dims = dims;
    a.q = reinterpret_cast<const __half *>(q);
    a.k_cache = reinterpret_cast<const __half *>(k_cache);
    a.v_cache = reinterpret_cast<const __half *>(v_cache);
    a.valid_len = valid_len;
    a.page_idx = nullptr;
    a.kpages = 0;
    a.scale = scale;
    a.out = reinterpret_cast<__half *>(out);
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return launch_attention(a, ctx);
}

int quest_append_kv(const gqaq_dims *dims, gqaq_half *k_cache, gqaq_half *v_cache, gqaq_half *meta,
                    const gqaq_half *k_new, const gqaq_half *v_new, const int32_t *pos, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(meta) || !aligned16(k_new) ||
        !aligned16(v_new) || !aligned16(pos))
        return GQAQ_ERR_INVALID_ARG;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    return launch_append_kv(dims, reinterpret_cast<__half *>(k_cache), reinterpret_cast<__half *>(v_cache),
                            reinterpret_cast<__half *>(meta), reinterpret_cast<const __half *>(k_new),
                            reinterpret_cast<const __half *>(v_new), pos, ctx);
}

int quest_update_meta(const gqaq_dims *dims, const gqaq_half *k_cache, const int32_t *valid_len,
                      gqaq_half *meta, int page_begin, int page_end, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(k_cache) || !aligned16(valid_len) || !aligned16(meta)) return GQAQ_ERR_INVALID_ARG;
    const int pmax = (dims->max_len + dims->page_size - 1) / dims->page_size;
    if (page_begin < 0 || page_end < page_begin || page_end > pmax) return GQAQ_ERR_INVALID_ARG;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    return launch_update_meta(dims, reinterpret_cast<const __half *>(k_cache), valid_len,
                              reinterpret_cast<__half *>(meta), page_begin, page_end, ctx);
}

int quest_score_pages(const gqaq_dims *dims, const gqaq_half *q, const gqaq_half *meta,
                      const int32_t *valid_len, float *scores, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(q) || !aligned16(meta) || !aligned16(valid_len) || !aligned16(scores))
        return GQAQ_ERR_INVALID_ARG;
    const int64_t pmax = (dims->max_len + dims->page_size - 1) / dims->page_size;
    if ((int64_t)dims->batch * dims->num_kv_heads * pmax > (int64_t)INT32_MAX - 1024) return GQAQ_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    return launch_score_pages(dims, reinterpret_cast<const __half *>(q), reinterpret_cast<const __half *>(meta),
                              valid_len, scores, ctx);
}

int quest_topk_pages(const gqaq_dims *dims, const float *scores, const int32_t *valid_len, int k,
                     int32_t *page_idx, void *workspace, size_t workspace_bytes, void *stream) {
    (void)workspace;
    (void)workspace_bytes;
    int rc = check_dims(dims, true);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(scores) || !aligned16(valid_len) || !aligned16(page_idx)) return GQAQ_ERR_INVALID_ARG;
    if (k < 1 || k > 65536) return GQAQ_ERR_INVALID_ARG;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    return launch_topk_pages(dims, scores, valid_len, k, page_idx, ctx);
}

int quest_sparse_attn(const gqaq_dims *dims, const gqaq_half *q, const gqaq_half *k_cache,
                      const gqaq_half *v_cache, const int32_t *valid_len, const int32_t *page_idx, int k,
                      float scale, gqaq_half *out, void *workspace, size_t workspace_bytes, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        !aligned16(valid_len) || !aligned16(page_idx))
        return GQAQ_ERR_INVALID_ARG;
    if (k < 1 || k > 65536) return GQAQ_ERR_INVALID_ARG;
    if (!isfinite(scale)) return GQAQ_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned16(workspace)) return GQAQ_ERR_WORKSPACE;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    if (k <= kFusedMaxPages) {
        // cluster kernel: attention and the log-sum-exp merge in one launch
        FusedArgs f = {};
        f.dims = dims;
        f.q = reinterpret_cast<const __half *>(q);
        f.k_cache = const_cast<__half *>(reinterpret_cast<const __half *>(k_cache));
        f.v_cache = const_cast<__half *>(reinterpret_cast<const __half *>(v_cache));
        f.meta = nullptr;
        f.valid_len = valid_len;
        f.page_idx = const_cast<int32_t *>(page_idx);
        f.kpages = k;
        f.scale = scale;
        f.out = reinterpret_cast<__half *>(out);
        return launch_quest_fused(f, ctx);
    }
    AttnArgs a = {};
    a.dims = dims;
    a.q = reinterpret_cast<const __half *>(q);
    a.k_cache = reinterpret_cast<const __half *>(k_cache);
    a.v_cache = reinterpret_cast<const __half *>(v_cache);
    a.valid_len = valid_len;
    a.page_idx = page_idx;
    a.kpages = k;
    a.scale = scale;
    a.out = reinterpret_cast<__half *>(out);
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return launch_attention(a, ctx);
}

int gqa_decode_attn_e4m3(const gqaq_dims *dims, const gqaq_half *q, const uint8_t *k_cache, const uint8_t *v_cache,
                         float k_scale, float v_scale, const int32_t *valid_len, float scale, gqaq_half *out,
                         void *workspace, size_t workspace_bytes, void *stream) {
    int rc = check_dims(dims, false);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(valid_len))
        return GQAQ_ERR_INVALID_ARG;
    if (!isfinite(scale) || !isfinite(k_scale) || !isfinite(v_scale)) return GQAQ_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned16(workspace)) return GQAQ_ERR_WORKSPACE;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    AttnArgs a = {};
    a.dims = dims;
    a.q = reinterpret_cast<const __half *>(q);
    a.k_cache = reinterpret_cast<const __half *>(k_cache);  // byte rows; typed as the kernels take it
    a.v_cache = reinterpret_cast<const __half *>(v_cache);
    a.valid_len = valid_len;
    a.page_idx = nullptr;
    a.kpages = 0;
    a.scale = scale;
    a.kv8 = true;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.out = reinterpret_cast<__half *>(out);
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return launch_attention(a, ctx);
}

int kv_append_e4m3(const gqaq_dims *dims, uint8_t *k_cache, uint8_t *v_cache, const gqaq_half *k_new,
                   const gqaq_half *v_new, const int32_t *pos, float k_inv_scale, float v_inv_scale, void *stream) {
    int rc = check_dims(dims, false);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(pos))
        return GQAQ_ERR_INVALID_ARG;
    if (!isfinite(k_inv_scale) || !isfinite(v_inv_scale)) return GQAQ_ERR_INVALID_ARG;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    return launch_append_e4m3(dims, k_cache, v_cache, reinterpret_cast<const __half *>(k_new),
                              reinterpret_cast<const __half *>(v_new), pos, k_inv_scale, v_inv_scale, ctx);
}

int quest_append_kv_e4m3(const gqaq_dims *dims, uint8_t *k_cache, uint8_t *v_cache, uint8_t *meta,
                         const gqaq_half *k_new, const gqaq_half *v_new, const int32_t *pos, float k_inv_scale,
                         float v_inv_scale, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(meta) || !aligned16(k_new) || !aligned16(v_new) ||
        !aligned16(pos))
        return GQAQ_ERR_INVALID_ARG;
    if (!isfinite(k_inv_scale) || !isfinite(v_inv_scale)) return GQAQ_ERR_INVALID_ARG;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    return launch_append_e4m3_meta(dims, k_cache, v_cache, meta, reinterpret_cast<const __half *>(k_new),
                                   reinterpret_cast<const __half *>(v_new), pos, k_inv_scale, v_inv_scale, ctx);
}

int quest_update_meta_e4m3(const gqaq_dims *dims, const uint8_t *k_cache, const int32_t *valid_len, uint8_t *meta,
                           int page_begin, int page_end, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(k_cache) || !aligned16(valid_len) || !aligned16(meta)) return GQAQ_ERR_INVALID_ARG;
    const int pmax = (dims->max_len + dims->page_size - 1) / dims->page_size;
    if (page_begin < 0 || page_end < page_begin || page_end > pmax) return GQAQ_ERR_INVALID_ARG;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    return launch_update_meta_e4m3(dims, k_cache, valid_len, meta, page_begin, page_end, ctx);
}

int quest_score_pages_e4m3(const gqaq_dims *dims, const gqaq_half *q, const uint8_t *meta, float k_scale,
                           const int32_t *valid_len, float *scores, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(q) || !aligned16(meta) || !aligned16(valid_len) || !aligned16(scores))
        return GQAQ_ERR_INVALID_ARG;
    if (!(isfinite(k_scale) && k_scale > 0.f)) return GQAQ_ERR_INVALID_ARG;  // a positive scale keeps the ranking
    const int64_t pmax = (dims->max_len + dims->page_size - 1) / dims->page_size;
    if ((int64_t)dims->batch * dims->num_kv_heads > 65535) return GQAQ_ERR_UNSUPPORTED;  // grid y
    if ((int64_t)dims->batch * dims->num_kv_heads * pmax > (int64_t)INT32_MAX - 1024) return GQAQ_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    return launch_score_pages_e4m3(dims, reinterpret_cast<const __half *>(q), meta, k_scale, valid_len, scores, ctx);
}

int quest_sparse_attn_e4m3(const gqaq_dims *dims, const gqaq_half *q, const uint8_t *k_cache, const uint8_t *v_cache,
                           float k_scale, float v_scale, const int32_t *valid_len, const int32_t *page_idx, int k,
                           float scale, gqaq_half *out, void *workspace, size_t workspace_bytes, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(valid_len) ||
        !aligned16(page_idx))
        return GQAQ_ERR_INVALID_ARG;
    if (k < 1 || k > 65536) return GQAQ_ERR_INVALID_ARG;
    if (!isfinite(scale) || !isfinite(k_scale) || !isfinite(v_scale)) return GQAQ_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned16(workspace)) return GQAQ_ERR_WORKSPACE;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    if (k <= kFusedMaxPages) {
        // cluster kernel: attention and the log-sum-exp merge in one launch
        FusedArgs f = {};
        f.dims = dims;
        f.q = reinterpret_cast<const __half *>(q);
        f.k_cache = const_cast<__half *>(reinterpret_cast<const __half *>(k_cache));
        f.v_cache = const_cast<__half *>(reinterpret_cast<const __half *>(v_cache));
        f.meta = nullptr;
        f.valid_len = valid_len;
        f.page_idx = const_cast<int32_t *>(page_idx);
        f.kpages = k;
        f.scale = scale;
        f.out = reinterpret_cast<__half *>(out);
        f.kv8 = true;
        f.k_scale = k_scale;
        f.v_scale = v_scale;
        return launch_quest_fused(f, ctx);
    }
    AttnArgs a = {};
    a.dims = dims;
    a.q = reinterpret_cast<const __half *>(q);
    a.k_cache = reinterpret_cast<const __half *>(k_cache);  // byte rows; typed as the kernels take it
    a.v_cache = reinterpret_cast<const __half *>(v_cache);
    a.valid_len = valid_len;
    a.page_idx = page_idx;
    a.kpages = k;
    a.scale = scale;
    a.kv8 = true;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.out = reinterpret_cast<__half *>(out);
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return launch_attention(a, ctx);
}

int quest_decode_attn_e4m3(const gqaq_dims *dims, const gqaq_half *q, uint8_t *k_cache, uint8_t *v_cache,
                           uint8_t *meta, const gqaq_half *k_new, const gqaq_half *v_new, const int32_t *pos,
                           float k_inv_scale, float v_inv_scale, float k_scale, float v_scale,
                           const int32_t *valid_len, int k, float scale, gqaq_half *out, float *scores,
                           int32_t *page_idx, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(meta) || !aligned16(valid_len) ||
        !aligned16(out))
        return GQAQ_ERR_INVALID_ARG;
    if (pos != nullptr && (!aligned16(pos) || !aligned16(k_new) || !aligned16(v_new))) return GQAQ_ERR_INVALID_ARG;
    if ((scores != nullptr && !aligned16(scores)) || (page_idx != nullptr && !aligned16(page_idx)))
        return GQAQ_ERR_INVALID_ARG;
    if (k < 1 || k > kFusedMaxPages) return k < 1 ? GQAQ_ERR_INVALID_ARG : GQAQ_ERR_UNSUPPORTED;
    if (!isfinite(scale) || !isfinite(v_scale) || !(isfinite(k_scale) && k_scale > 0.f)) return GQAQ_ERR_INVALID_ARG;
    if (pos != nullptr && (!isfinite(k_inv_scale) || !isfinite(v_inv_scale))) return GQAQ_ERR_INVALID_ARG;
    const int64_t pmax = (dims->max_len + dims->page_size - 1) / dims->page_size;
    if ((int64_t)dims->batch * dims->num_kv_heads * pmax > (int64_t)INT32_MAX - 1024) return GQAQ_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    if (ctx.quest_kernel == 2) return GQAQ_ERR_UNSUPPORTED;  // the work-queue kernel reads fp16 caches only
    FusedArgs f = {};
    f.dims = dims;
    f.q = reinterpret_cast<const __half *>(q);
    f.k_cache = reinterpret_cast<__half *>(k_cache);  // byte rows; typed as the kernels take them
    f.v_cache = reinterpret_cast<__half *>(v_cache);
    f.meta = reinterpret_cast<__half *>(meta);
    f.k_new = reinterpret_cast<const __half *>(k_new);
    f.v_new = reinterpret_cast<const __half *>(v_new);
    f.pos = pos;
    f.valid_len = valid_len;
    f.page_idx = page_idx;
    f.scores = scores;
    f.kpages = k;
    f.scale = scale;
    f.out = reinterpret_cast<__half *>(out);
    f.kv8 = true;
    f.k_inv = k_inv_scale;
    f.v_inv = v_inv_scale;
    f.k_scale = k_scale;
    f.v_scale = v_scale;
    return launch_quest_fused(f, ctx);
}

int gqa_decode_attn_int4(const gqaq_dims *dims, const gqaq_half *q, const uint8_t *k_codes, const float *k_scales,
                         const uint8_t *v_codes, const float *v_scales, const int32_t *valid_len, float scale,
                         gqaq_half *out, void *workspace, size_t workspace_bytes, void *stream) {
    int rc = check_dims(dims, false);
    if (rc != GQAQ_OK) return rc;
    if (dims->max_len % 4 != 0) return GQAQ_ERR_UNSUPPORTED;  // scale rows are 16-byte multiples
    if (!aligned16(q) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scales) ||
        !aligned16(v_scales) || !aligned16(out) || !aligned16(valid_len))
        return GQAQ_ERR_INVALID_ARG;
    if (!isfinite(scale)) return GQAQ_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned16(workspace)) return GQAQ_ERR_WORKSPACE;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    AttnArgs a = {};
    a.dims = dims;
    a.q = reinterpret_cast<const __half *>(q);
    a.k_cache = reinterpret_cast<const __half *>(k_codes);  // byte rows; typed as the kernels take it
    a.v_cache = reinterpret_cast<const __half *>(v_codes);
    a.valid_len = valid_len;
    a.scale = scale;
    a.kv4 = true;
    a.k_scales = k_scales;
    a.v_scales = v_scales;
    a.out = reinterpret_cast<__half *>(out);
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return launch_attention(a, ctx);
}

int kv_append_int4(const gqaq_dims *dims, uint8_t *k_codes, float *k_scales, uint8_t *v_codes, float *v_scales,
                   const gqaq_half *k_new, const gqaq_half *v_new, const int32_t *pos, void *stream) {
    int rc = check_dims(dims, false);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scales) || !aligned16(v_scales) ||
        !aligned16(k_new) || !aligned16(v_new) || !aligned16(pos))
        return GQAQ_ERR_INVALID_ARG;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    return launch_append_int4(dims, k_codes, k_scales, v_codes, v_scales, reinterpret_cast<const __half *>(k_new),
                              reinterpret_cast<const __half *>(v_new), pos, ctx);
}

namespace {
int check_prefill(const gqaq_dims *dims, int q_len) {
    const int rc = check_dims(dims, false);
    if (rc != GQAQ_OK) return rc;
    if (q_len < 1 || q_len > dims->max_len) return GQAQ_ERR_INVALID_ARG;
    const int64_t qrows = (int64_t)dims->batch * dims->num_q_heads * q_len;
    if (qrows > (int64_t)INT32_MAX / 128) return GQAQ_ERR_UNSUPPORTED;
    return GQAQ_OK;
}
}  // namespace

size_t gqaq_prefill_workspace_bytes(const gqaq_dims *dims, int q_len) {
    if (check_prefill(dims, q_len) != GQAQ_OK) return 0;
    LaunchCtx ctx;
    if (make_ctx(&ctx, nullptr) != GQAQ_OK) return 0;
    return prefill_workspace_bytes(dims, q_len, ctx);
}

int gqa_prefill_attn(const gqaq_dims *dims, int q_len, const gqaq_half *q, const gqaq_half *k_cache,
                     const gqaq_half *v_cache, const int32_t *start, float scale, gqaq_half *out, void *workspace,
                     size_t workspace_bytes, void *stream) {
    int rc = check_prefill(dims, q_len);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(start))
        return GQAQ_ERR_INVALID_ARG;
    if (!isfinite(scale)) return GQAQ_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned16(workspace)) return GQAQ_ERR_WORKSPACE;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    PrefillArgs a;
    a.dims = dims;
    a.q_len = q_len;
    a.q = reinterpret_cast<const __half *>(q);
    a.k_cache = reinterpret_cast<const __half *>(k_cache);
    a.v_cache = reinterpret_cast<const __half *>(v_cache);
    a.start = start;
    a.scale = scale;
    a.out = reinterpret_cast<__half *>(out);
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return launch_prefill(a, ctx);
}

int quest_decode_attn(const gqaq_dims *dims, const gqaq_half *q, gqaq_half *k_cache, gqaq_half *v_cache,
                      gqaq_half *meta, const gqaq_half *k_new, const gqaq_half *v_new, const int32_t *pos,
                      const int32_t *valid_len, int k, float scale, gqaq_half *out, float *scores,
                      int32_t *page_idx, void *workspace, size_t workspace_bytes, void *stream) {
    int rc = check_dims(dims, true);
    if (rc != GQAQ_OK) return rc;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(meta) ||
        !aligned16(valid_len) || !aligned16(out))
        return GQAQ_ERR_INVALID_ARG;
    if (pos != nullptr && (!aligned16(pos) || !aligned16(k_new) || !aligned16(v_new))) return GQAQ_ERR_INVALID_ARG;
    if ((scores != nullptr && !aligned16(scores)) || (page_idx != nullptr && !aligned16(page_idx)))
        return GQAQ_ERR_INVALID_ARG;
    if (k < 1 || k > 65536) return GQAQ_ERR_INVALID_ARG;
    if (workspace != nullptr && !aligned16(workspace)) return GQAQ_ERR_WORKSPACE;
    if (!isfinite(scale)) return GQAQ_ERR_INVALID_ARG;
    const int64_t pmax = (dims->max_len + dims->page_size - 1) / dims->page_size;
    if ((int64_t)dims->batch * dims->num_kv_heads * pmax > (int64_t)INT32_MAX - 1024) return GQAQ_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    rc = make_ctx(&ctx, stream);
    if (rc != GQAQ_OK) return rc;
    FusedArgs f = {};
    f.dims = dims;
    f.q = reinterpret_cast<const __half *>(q);
    f.k_cache = reinterpret_cast<__half *>(k_cache);
    f.v_cache = reinterpret_cast<__half *>(v_cache);
    f.meta = reinterpret_cast<__half *>(meta);
    f.k_new = reinterpret_cast<const __half *>(k_new);
    f.v_new = reinterpret_cast<const __half *>(v_new);
    f.pos = pos;
    f.valid_len = valid_len;
    f.page_idx = page_idx;
    f.scores = scores;
    f.kpages = k;
    f.scale = scale;
    f.out = reinterpret_cast<__half *>(out);
    f.workspace = workspace;
    f.workspace_bytes = workspace_bytes;
    // The cluster kernel when it covers the shape (the faster one at every
    // measured shape); the work-queue kernel for larger k, or when forced.
    const bool queue_ok = workspace != nullptr && quest_stream_workspace_bytes(dims, k, ctx) > 0;
    const bool cluster_ok = k <= kFusedMaxPages;
    if (ctx.quest_kernel == 2 || (ctx.quest_kernel == 0 && !cluster_ok)) {
        if (!queue_ok) return workspace == nullptr ? GQAQ_ERR_WORKSPACE : GQAQ_ERR_UNSUPPORTED;
        return launch_quest_stream(f, ctx);
    }
    if (!cluster_ok) return GQAQ_ERR_UNSUPPORTED;
    return launch_quest_fused(f, ctx);
}

}  // extern "C"
