// Shared pieces of the persistent (TMA-pipelined) kernels: bounded mbarrier
// waits, bit packing of carries into shared-memory slots, and the host-side
// tensor-map encoder.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "sc_device.cuh"
#include "sc_tma.cuh"

namespace scg {
namespace persist {

template <class V>
__device__ __forceinline__ unsigned long long pack_bits(V v) {
    if constexpr (sizeof(V) == 4) return to_bits32(v);
    else return to_bits64(v);
}
template <class V>
__device__ __forceinline__ V unpack_bits(unsigned long long b) {
    V v;
    if constexpr (sizeof(V) == 4) from_bits32((uint32_t)b, v);
    else from_bits64(b, v);
    return v;
}

// Longest sleep of one probe in the bounded waits below.  A waiter wakes as
// soon as its phase completes; the bound only delays noticing *end_k and the
// time limit.
constexpr uint32_t kWaitSuspendNs = 1000;

// Bounded wait on an mbarrier phase: gives up (false) after `limit_ns`, or
// as soon as *end_k (when given) is <= k (iteration k will never come).
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns,
                                         const volatile int* end_k = nullptr, int k = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (unsigned i = 1; i < (1u << 30); ++i) {
        if (mbar_try_wait_sleep(bar, parity, kWaitSuspendNs)) return true;
        if (end_k && *end_k <= k) return false;
        if ((i & 3u) == 0 && global_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Warp-uniform variant: lane 0 waits, the verdict is broadcast, and every
// lane then observes the completed phase itself (so each lane's later reads of
// what the phase protects are ordered after it).
__device__ __forceinline__ bool warp_bar_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns,
                                              const volatile int* end_k = nullptr, int k = 0) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;  // usually already complete
    bool good = true;
    if ((threadIdx.x & 31) == 0) good = bar_wait(bar, parity, limit_ns, end_k, k);
    good = __shfl_sync(0xffffffffu, good, 0);
    if (good) good = mbar_try_wait(bar, parity);
    return __all_sync(0xffffffffu, good);
}

__device__ __forceinline__ int vload(const int* p) { return *reinterpret_cast<const volatile int*>(p); }
__device__ __forceinline__ void vstore(int* p, int v) { *reinterpret_cast<volatile int*>(p) = v; }

// ------------------------------------------------------------- host side
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn_ptr = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn_ptr = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    return fn_ptr;
}

// The first `rows` rows of 128 bytes at `base`, boxes of `box_rows` rows,
// 128-byte swizzle.  `base` must be 16-byte aligned.
inline bool make_map(CUtensorMap* m, const void* base, unsigned long long rows, unsigned box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {32, rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Chunk ids of a persistent kernel, taken by its producer thread from the
// launch's monotone counter.  Far from the end each id is requested one chunk
// ahead of use, which hides the atomic's latency; within the last `margin`
// chunks (a round of the grid) an id is requested only when it is needed, so
// the last chunks go to CTAs that are free instead of to CTAs that reserved
// them while still busy (measured on GB300 the same as requesting every id
// ahead: the CTAs' end times spread over about two chunks either way).  A CTA
// stops at its first id >= num_chunks and requests
// none after it, so a launch advances the counter by exactly num_chunks +
// grid, which the host adds to the base for the next launch (the counter must
// start every launch at the base: an id below it would name a negative chunk,
// which take() turns into an error and the end of the CTA's work).
struct ChunkIds {
    unsigned long long* ctr;
    unsigned long long base;
    long long num_chunks, margin;
    unsigned int* err;
    unsigned long long next = 0;
    bool have = false;
    __device__ __forceinline__ void start() {
        next = atomicAdd(ctr, 1ull);
        have = true;
    }
    __device__ __forceinline__ long long take() {
        if (!have) next = atomicAdd(ctr, 1ull);
        long long c = (long long)(next - base);
        have = false;
        if (c < 0) {  // the counter is behind the host's base: never use the id
            atomicCAS(err, 0u, (unsigned)DEV_INTERNAL);
            return num_chunks;
        }
        if (c + margin < num_chunks) {
            next = atomicAdd(ctr, 1ull);
            have = true;
        }
        return c;
    }
};

// Opt a kernel in to more than 48 KiB of dynamic shared memory, once per device.
template <class K>
inline cudaError_t allow_smem(K kernel, int bytes, std::atomic<unsigned long long>& done_mask) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done_mask.load() & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done_mask.fetch_or(bit);
    return e;
}

}  // namespace persist
}  // namespace scg
