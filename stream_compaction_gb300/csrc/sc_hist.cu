// Histogram of int32 bin indices, the counting step of "histogram + exclusive
// scan" ("Chapter 9 Parallel Patterns: Prefix Sum - Scan Algorithms", PMPP
// notes, section 4.2: a radix sort's digit pass scans the digit histogram to
// find where each bucket starts; converting a sparse matrix from COO to CSR
// scans the per-row counts to get the row offsets).  The scan is the library's
// int64 single-pass scan (sc_api.cu).
//
// counts[b] += number of i with bins[i] == b, 0 <= b < nbins (entries outside
// are skipped).  Beyond kWarpCopyBins bins, a run of equal neighbouring bins
// in a warp step (512 consecutive entries, 16 per thread) is counted with one
// atomic, so sorted input (CSR rows) costs about one atomic per row per warp
// step.  Up to
// kWarpCopyBins bins each warp counts into its own
// shared-memory histogram (plain shared atomics), up to kSmemBins bins each CTA
// into one shared histogram; the CTA adds its counts to the global ones once
// at the end.  Beyond that the atomics go to the global counts directly.
#include <algorithm>

#include "sc_launch.h"

namespace scg {

namespace {

constexpr int kHistThreads = 512;

// kMode: 0 global atomics (one per run of equal neighbours), 1 one shared
// histogram per CTA (likewise), 2 one shared histogram per warp (plain shared
// atomics: contention stays inside the warp; for small bin counts).
template <int kMode>
__global__ void __launch_bounds__(kHistThreads) histogram_kernel(const int32_t* __restrict__ bins, long long n,
                                                                 int nbins, unsigned long long* __restrict__ counts,
                                                                 int vec) {
    extern __shared__ unsigned int sh[];
    const int lane = threadIdx.x & 31;
    constexpr int kWarps = kHistThreads / 32;
    const int copies = kMode == 2 ? kWarps : 1;
    if constexpr (kMode != 0) {
        for (int b = threadIdx.x; b < nbins * copies; b += blockDim.x) sh[b] = 0u;
        __syncthreads();
    }
    unsigned int* const mine = sh + (kMode == 2 ? (threadIdx.x >> 5) * nbins : 0);
    auto add = [&](int b) {  // one shared histogram per warp: plain shared atomics
        if (b >= 0 && b < nbins) atomicAdd(&mine[b], 1u);
    };
    if constexpr (kMode != 2) {
        // Runs of equal neighbours, 16 consecutive bins per thread (a warp step
        // covers 512): the thread counts its own runs; a run that reaches the
        // thread's end continues into the next lanes' first runs, whose lengths
        // a reverse scan over the warp gathers, so each run in the warp step
        // costs one atomic (a run that crosses warp steps costs one per step).
        constexpr int kPer = 16;
        auto emit = [&](int b, unsigned len) {
            if (b >= 0 && b < nbins) {
                if constexpr (kMode == 1) atomicAdd(&sh[b], len);
                else atomicAdd(&counts[b], (unsigned long long)len);
            }
        };
        auto step = [&](const int (&v)[kPer]) {
            const int prev = __shfl_up_sync(0xffffffffu, v[kPer - 1], 1);
            uint32_t hm = (lane == 0 || v[0] != prev) ? 1u : 0u;  // bit k: a run starts at item k
#pragma unroll
            for (int k = 1; k < kPer; ++k) hm |= (v[k] != v[k - 1] ? 1u : 0u) << k;
            // (c, w): this lane's leading continuation length, and whether the
            // whole lane continues the run before it; the suffix composition
            // x -> c + w * x over the later lanes gives the length a run
            // reaching this lane's end gains from them
            unsigned c = hm & 1u ? 0u : (hm ? (unsigned)(__ffs(hm) - 1) : (unsigned)kPer);
            bool w = hm == 0u;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const unsigned c2 = __shfl_down_sync(0xffffffffu, c, d);
                const bool w2 = __shfl_down_sync(0xffffffffu, (unsigned)w, d) != 0u;
                if (lane + d < 32) {
                    if (w) c += c2;
                    w = w && w2;
                }
            }
            const unsigned after = __shfl_down_sync(0xffffffffu, c, 1);  // every lane takes part
            const unsigned gain = lane == 31 ? 0u : after;
            // this lane's runs, last first: the last one gains the later lanes' continuation
            unsigned end = kPer + gain;
#pragma unroll
            for (int k = kPer - 1; k >= 0; --k) {
                if ((hm >> k) & 1u) {
                    emit(v[k], end - (unsigned)k);
                    end = (unsigned)k;
                }
            }
        };
        constexpr int kSteps = 2;  // warp steps per loop iteration, all loads first
        const long long nchunks = (n + kPer - 1) / kPer;  // per-thread chunks of 16 bins
        const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
        const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
        for (long long c0 = wid * 32 * kSteps; c0 < nchunks; c0 += nwarps * 32 * kSteps) {
            int v[kSteps][kPer];
#pragma unroll
            for (int u = 0; u < kSteps; ++u) {
                const long long i = (c0 + u * 32 + lane) * kPer;
                if (vec && i + kPer <= n) {
#pragma unroll
                    for (int q = 0; q < kPer / 4; ++q) {
                        const int4 r = __ldg(reinterpret_cast<const int4*>(bins + i) + q);
                        v[u][4 * q] = r.x; v[u][4 * q + 1] = r.y; v[u][4 * q + 2] = r.z; v[u][4 * q + 3] = r.w;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < kPer; ++k) v[u][k] = i + k < n ? __ldg(bins + i + k) : -1;
                }
            }
#pragma unroll
            for (int u = 0; u < kSteps; ++u) step(v[u]);
        }
        if constexpr (kMode == 1) {
            __syncthreads();
            for (int b = threadIdx.x; b < nbins; b += blockDim.x)
                if (sh[b]) atomicAdd(&counts[b], (unsigned long long)sh[b]);
        }
        return;
    }
    // kMode 2: groups of 4 consecutive bins (16-byte loads when aligned),
    // kUnroll warp steps of 32 groups per loop iteration with all loads issued
    // first
    constexpr int kUnroll = 4;
    const long long ngroups = (n + 3) / 4;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long g0 = wid * 32 * kUnroll; g0 < ngroups; g0 += nwarps * 32 * kUnroll) {
        int v[kUnroll][4];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long g = g0 + u * 32 + lane;
            v[u][0] = v[u][1] = v[u][2] = v[u][3] = -1;
            if (g < ngroups) {
                const long long i = g * 4;
                if (vec && i + 4 <= n) {
                    const int4 q = __ldg(reinterpret_cast<const int4*>(bins) + g);
                    v[u][0] = q.x; v[u][1] = q.y; v[u][2] = q.z; v[u][3] = q.w;
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (i + k < n) v[u][k] = __ldg(bins + i + k);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
            for (int k = 0; k < 4; ++k) add(v[u][k]);
    }
    __syncthreads();
    for (int b = threadIdx.x; b < nbins; b += blockDim.x) {
        unsigned long long c = 0;
        for (int w = 0; w < copies; ++w) c += sh[w * nbins + b];
        if (c) atomicAdd(&counts[b], c);
    }
}

}  // namespace

constexpr int kSmemBins = 32768;      // one shared histogram per CTA up to here (128 KiB)
constexpr int kWarpCopyBins = 1024;   // one shared histogram per warp up to here (16 x 4 KiB)

template <int kMode>
cudaError_t launch_mode(const int32_t* bins, long long n, int nbins, unsigned long long* counts, unsigned grid,
                        int smem, int vec, cudaStream_t s) {
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(histogram_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    histogram_kernel<kMode><<<grid, kHistThreads, smem, s>>>(bins, n, nbins, counts, vec);
    return cudaGetLastError();
}

cudaError_t launch_histogram(const int32_t* bins, long long n, int nbins, unsigned long long* counts, int num_sms,
                             cudaStream_t s) {
    const int vec = (reinterpret_cast<uintptr_t>(bins) % 16) == 0;
    const long long ngroups = (n + 3) / 4;
    // CTAs with at least one warp iteration each (kUnroll warp steps of 32 groups)
    auto grid_of = [&](int per_sm, int unroll) {
        const long long want = (ngroups + 32 * unroll - 1) / (32 * unroll) * 32 / kHistThreads + 1;
        return (unsigned)std::max<long long>(1, std::min<long long>(want, (long long)num_sms * per_sm));
    };
    // shared histograms: a few CTAs per SM, each flush costs nbins atomics;
    // the run-counting modes cover 1024 bins (256 groups) per warp iteration
    if (nbins <= kWarpCopyBins)
        return launch_mode<2>(bins, n, nbins, counts, grid_of(2, 4), nbins * 4 * (kHistThreads / 32), vec, s);
    if (nbins <= kSmemBins)
        return launch_mode<1>(bins, n, nbins, counts, grid_of(nbins <= 8192 ? 2 : 1, 8), nbins * 4, vec, s);
    return launch_mode<0>(bins, n, nbins, counts, grid_of(2, 8), 0, vec, s);
}

}  // namespace scg
