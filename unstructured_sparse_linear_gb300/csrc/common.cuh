// Shared device helpers for the spops GB300 kernels: element types, 16-byte vector
// load/store with fp32 widening, bounded mbarrier waits and the device error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spops {

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Error codes a kernel may record in the device error word (first writer wins).
enum DeviceError : int {
    kDevErrNone = 0,
    kDevErrMbarTimeout = 1,      // an mbarrier wait ran past its time limit
    kDevErrRowOffsets = 2,       // row_offsets not non-decreasing / wrong ends
    kDevErrColRange = 3,         // a column index outside [0, n)
    kDevErrColOrder = 4,         // columns not strictly increasing inside a row
    kDevErrRowIdxPerm = 5,       // row_idx is not a permutation of 0..m-1
    kDevErrTmemAlloc = 6,        // tensor-memory allocation returned an unusable address
};

__device__ __forceinline__ void record_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ------------------------------------------------------------------ element types

template <typename T>
struct Elt;

template <>
struct Elt<float> {
    static constexpr int kVec = 4;  // elements per 16-byte vector
    __device__ __forceinline__ static float to_f(float x) { return x; }
    __device__ __forceinline__ static float from_f(float x) { return x; }
    __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

template <>
struct Elt<__half> {
    static constexpr int kVec = 8;
    __device__ __forceinline__ static float to_f(__half x) { return __half2float(x); }
    __device__ __forceinline__ static __half from_f(float x) { return __float2half_rn(x); }
    __device__ __forceinline__ static float2 h2(uint32_t u) {
        __half2 h = *reinterpret_cast<__half2*>(&u);
        return __half22float2(h);
    }
    __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
        float2 a = h2(v.x), b = h2(v.y), c = h2(v.z), d = h2(v.w);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    }
    __device__ __forceinline__ static uint32_t p2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(p2(f[0], f[1]), p2(f[2], f[3]), p2(f[4], f[5]), p2(f[6], f[7]));
    }
};

template <>
struct Elt<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ __forceinline__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ __forceinline__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
    // bf16 is the upper half of an fp32 bit pattern, so widening is a shift (exact).
    __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
        f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
        f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
        f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xffff0000u);
        f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t p2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(p2(f[0], f[1]), p2(f[2], f[3]), p2(f[4], f[5]), p2(f[6], f[7]));
    }
};

// Index lists: int16 lists are read as unsigned 16-bit so that 0..32767 and any stray
// negative pattern both land in 0..65535 (callers guarantee indices < 32768).
template <typename I>
__device__ __forceinline__ int idx_of(I x) {
    return static_cast<int>(x);
}

// ------------------------------------------------------------------ loads

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_v4(const void* p) {
    return *reinterpret_cast<const uint4*>(p);
}

// ------------------------------------------------------------------ shared memory / mbarrier

// Barrier `id` (1 .. 15; 0 is __syncthreads) over the first nthreads threads of the CTA
// (a multiple of 32; every one of them must arrive).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// named_barrier that also ANDs pred over the arriving threads (all of them get the result).
__device__ __forceinline__ bool named_barrier_and(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Invalidate an idle mbarrier (every phase consumed, nothing pending) before re-initializing it.
__device__ __forceinline__ void mbar_inval(uint32_t bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait until the mbarrier phase with the given parity completes. Gives up after about
// limit_ns of wall time (kMbarTimeoutNs in mbar_wait), records kDevErrMbarTimeout and
// returns false; the time is read every 256 polls.
constexpr uint64_t kMbarTimeoutNs = 2000000000ull;  // 2 s
constexpr uint32_t kMbarPollNs = 64;                 // suspend-time hint of one poll

__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, int* err, uint64_t limit_ns) {
    uint32_t done = 0;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        // a short suspend-time hint: the thread re-polls within ~kMbarPollNs instead of staying
        // suspended for the (longer) system-dependent limit, so a pipeline stage hands over
        // promptly
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity), "n"(kMbarPollNs)
            : "memory");
        if (done) return true;
        if ((it & 255u) == 0) {
            uint64_t t = global_timer_ns();
            if (it == 0) t0 = t;
            else if (t - t0 > limit_ns) {
                record_error(err, kDevErrMbarTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err) {
    return mbar_wait_for(bar, parity, err, kMbarTimeoutNs);
}

// 1-D bulk async copies (TMA engine, no tensor map): global -> shared with mbarrier
// completion, shared -> global tracked by bulk groups. Addresses 16-byte aligned, sizes
// multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ panel skip flags

// Per-panel skip flags (panels of 128 row_idx positions handled on the tensor cores) as the
// general row kernels read them: copied into shared memory once per CTA when there are at
// most kSkipCache panels, so the many tests of a persistent loop are not global loads.
constexpr int kSkipCache = 4096;

struct SkipFlags {
    const uint8_t* f;  // the shared copy or the global flags (generic address); nullptr: none
    bool all;          // every panel is skipped (known when the flags are cached)
    __device__ __forceinline__ bool operator()(int64_t pos) const { return f && f[pos >> 7] != 0; }
};

// Call after pdl_wait (the flags come from the plan), by every thread of the CTA.
__device__ __forceinline__ SkipFlags load_skip_flags(const uint8_t* skip, int64_t m, uint8_t* cache) {
    const int64_t P = (m + 127) >> 7;
    const bool cached = skip != nullptr && P <= kSkipCache;
    int open = 0;  // this thread saw a panel that is not skipped
    if (cached)
        for (int64_t i = threadIdx.x; i < P; i += blockDim.x) {
            cache[i] = skip[i];
            open |= skip[i] == 0;
        }
    const bool any_open = __syncthreads_or(open) != 0;
    return SkipFlags{cached ? cache : skip, cached && !any_open};
}

// ------------------------------------------------------------------ thread-block clusters

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster arrives; shared-memory writes before it are
// visible to the cluster's reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address in CTA `rank`'s shared memory of the local shared address `addr`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, int rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(addr), "r"(rank));
    return ra;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_cluster_f4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_shared_f4(uint32_t addr, float4 v) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// Programmatic dependent launch (kernels launched with launch_pdl): pdl_trigger lets the
// next kernel in the stream begin launching; pdl_wait blocks until the previous kernel has
// finished and its writes are visible. Both do nothing for an ordinary launch.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace spops
