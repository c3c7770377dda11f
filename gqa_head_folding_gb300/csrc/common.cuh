// common.cuh -- sm_103a building blocks shared by the kernels: mbarriers with
// bounded waits, TMA tile loads, named barriers, and the balanced partition
// of work tiles over a persistent grid.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/gqaq.h"

namespace gqaq {

// ---------------------------------------------------------------------------
// Options and per-launch context (host side fills it)
// ---------------------------------------------------------------------------
struct LaunchCtx {
    cudaStream_t stream;
    int device;
    int num_sms;
    int max_ctas;          // 0 = automatic
    uint64_t timeout_ns;   // bound on every in-kernel wait
    int test_stall;        // attention producer issues nothing (timeout test)
    int cluster_size;      // fused Quest kernel: forced CTAs per cluster, 0 = automatic
    int pdl;               // launch with programmatic stream serialization
    int quest_kernel;      // fused Quest kernel: 0 automatic, 1 cluster, 2 work queue
    int prefill_splits;    // prefill context splits per item: 0 automatic, n forced
    int prefill_kernel;    // prefill kernel: 0 automatic (tensor memory), 1 tensor memory, 2 warp MMA
    int quest_early_meta;  // fused Quest kernel: first metadata tiles read before the grid dependency wait
    int dense_early_kv;    // dense attention: first K/V tiles read before the grid dependency wait
    int *status;           // device status word
};

// ---------------------------------------------------------------------------
// Small PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// One probe of the phase with parity `parity`; the hardware may suspend the
// thread for up to ~20 us while the phase is pending.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// One probe that may suspend the thread for up to about `ns` nanoseconds
// while the phase is pending (for a thread that watches several barriers).
__device__ __forceinline__ bool mbar_try_wait_ns(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with parity `parity`. Returns false when
// `timeout_ns` elapsed or `*abort` became nonzero first.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                          const volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort != nullptr && *abort) return false;
        if (global_timer_ns() - t0 >= timeout_ns) return false;
    }
}

// 2-D TMA tile load global -> shared, completion signalled on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t x,
                                            int32_t y, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// 3-D TMA tile load global -> shared, completion signalled on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// acc + (lo or hi half of a) * (lo or hi half of b), fp16 inputs, fp32 FMA.
// The product of two fp16 values is exact in fp32; one rounding per step.
__device__ __forceinline__ float fma_h_lo(uint32_t a, uint32_t b, float acc) {
    float r;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %3;\n\t}"
        : "=f"(r)
        : "r"(a), "r"(b), "f"(acc));
    return r;
}
__device__ __forceinline__ float fma_h_hi(uint32_t a, uint32_t b, float acc) {
    float r;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, %3;\n\t}"
        : "=f"(r)
        : "r"(a), "r"(b), "f"(acc));
    return r;
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t bits) {
    __half2 h = *reinterpret_cast<__half2 *>(&bits);
    return __half22float2(h);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel in the stream is still
// running. It must wait here before touching global memory that the previous
// kernel writes or reads. It lets its own dependents launch at once: they
// wait in the same way for this grid to finish.
__device__ __forceinline__ void pdl_wait_and_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Atomic add at gpu scope with acquire-release semantics: it publishes the
// writes that happen before it (including other threads' writes ordered by a
// CTA barrier) and makes visible the writes released by earlier adds.
__device__ __forceinline__ unsigned atomic_add_acq_rel_gpu(unsigned *ptr, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void raise_flag(int *status, int flag) {
    if (status != nullptr) atomicOr(status, flag);
}

// Host: launch `kern` on ctx.stream, optionally as a cluster of `cluster`
// CTAs, with programmatic stream serialization when ctx.pdl is set.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, const LaunchCtx &ctx,
                                 int cluster, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute at[2];
    int n = 0;
    if (cluster > 0) {
        at[n].id = cudaLaunchAttributeClusterDimension;
        at[n].val.clusterDim.x = (unsigned)cluster;
        at[n].val.clusterDim.y = 1;
        at[n].val.clusterDim.z = 1;
        ++n;
    }
    if (ctx.pdl) {
        at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = at;
    cfg.numAttrs = (unsigned)n;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// Balanced partition: T work tiles over `grid` persistent CTAs.
// CTA c owns tiles [floor(c*T/grid), floor((c+1)*T/grid)).
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int64_t tile_begin(int64_t c, int64_t T, int64_t grid) {
    return (c * T) / grid;
}
// The CTA whose (non-empty) range contains tile t (0 <= t < T).
__host__ __device__ __forceinline__ int64_t tile_owner(int64_t t, int64_t T, int64_t grid) {
    return ((t + 1) * grid - 1) / T;
}

__device__ __forceinline__ int clamp_len(int v, int lmax) {
    return v < 0 ? 0 : (v > lmax ? lmax : v);
}

// Work tiles of one (sequence, KV head) unit.
//  dense : ceil(len / tile_tokens) tiles of consecutive tokens
//  sparse: ceil(min(k, ceil(len / S)) / pages_per_tile) tiles of selected pages
struct TileRule {
    int sparse;
    int lmax;
    int page_size;
    int kpages;
    int tile_tokens;     // dense
    int pages_per_tile;  // sparse
    __device__ __forceinline__ int tiles(int raw_len) const {
        const int len = clamp_len(raw_len, lmax);
        if (!sparse) return (len + tile_tokens - 1) / tile_tokens;
        const int P = (len + page_size - 1) / page_size;
        const int nsel = P < kpages ? P : kpages;
        return (nsel + pages_per_tile - 1) / pages_per_tile;
    }
};

// Whole warp: total tiles T over all units, and (when t_target < T) the
// sequence b holding tile t_target plus the tile offset of b's first unit.
__device__ __forceinline__ void locate_tile(const int *valid_len, int B, int Hkv, const TileRule &rule,
                                            int64_t t_target, int64_t &T_out, int &b_out,
                                            int64_t &off_out) {
    const int lane = threadIdx.x & 31;
    int64_t cum = 0;
    b_out = -1;
    off_out = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
        const int b = b0 + lane;
        const int64_t n = (b < B) ? (int64_t)Hkv * rule.tiles(valid_len[b]) : 0;
        int64_t incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int64_t total = __shfl_sync(0xffffffffu, incl, 31);
        const unsigned hit = __ballot_sync(0xffffffffu, (b < B) && (cum + incl > t_target));
        if (b_out < 0 && hit != 0u) {  // warp-uniform branch
            const int src = __ffs(hit) - 1;
            const int64_t excl = __shfl_sync(0xffffffffu, incl - n, src);
            b_out = b0 + src;
            off_out = cum + excl;
        }
        cum += total;
    }
    T_out = cum;
}

}  // namespace gqaq
