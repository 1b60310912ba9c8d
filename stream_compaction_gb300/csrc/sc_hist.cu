// Histogram of int32 bin indices, the counting step of "histogram + exclusive
// scan" ("Chapter 9 Parallel Patterns: Prefix Sum - Scan Algorithms", PMPP
// notes, section 4.2: a radix sort's digit pass scans the digit histogram to
// find where each bucket starts; converting a sparse matrix from COO to CSR
// scans the per-row counts to get the row offsets).  The scan is the library's
// int64 single-pass scan (sc_api.cu).
//
// counts[b] += number of i with bins[i] == b, 0 <= b < nbins (entries outside
// are skipped).  Beyond kWarpCopyBins bins, a run of equal neighbouring bins
// in a warp step (128 consecutive entries) is counted with one atomic, so
// sorted input (CSR rows) costs about one atomic per row per warp step.  Up to
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
    // The warp step's 128 bins in memory order (lane l holds 4l .. 4l+3): one
    // atomic per run of equal neighbours, its length from the next run's start
    // (a shuffle finds the starts, a ballot and one shuffle the next start in
    // a later lane).  No __match_any_sync: its cost grows with the number of
    // distinct values and it bounded this kernel (address-divergence unit 90 %
    // busy on CSR rows).
    auto add_runs = [&](const int (&b)[4]) {
        const int prev = __shfl_up_sync(0xffffffffu, b[3], 1);
        bool h[4];
        h[0] = lane == 0 || b[0] != prev;
#pragma unroll
        for (int k = 1; k < 4; ++k) h[k] = b[k] != b[k - 1];
        const int fh = h[0] ? 0 : h[1] ? 1 : h[2] ? 2 : h[3] ? 3 : 4;  // first run start in this lane
        const unsigned any = __ballot_sync(0xffffffffu, fh < 4);
        const unsigned later = lane == 31 ? 0u : any & (0xffffffffu << (lane + 1));
        const int nl = later ? __ffs(later) - 1 : 32;
        const int nfh = __shfl_sync(0xffffffffu, fh, nl & 31);
        int end = nl < 32 ? 4 * nl + nfh : 128;  // start of the run after this lane's last
#pragma unroll
        for (int k = 3; k >= 0; --k) {
            if (h[k]) {
                const int pos = 4 * lane + k;
                if (b[k] >= 0 && b[k] < nbins) {
                    if constexpr (kMode == 1) atomicAdd(&sh[b[k]], (unsigned)(end - pos));
                    else atomicAdd(&counts[b[k]], (unsigned long long)(end - pos));
                }
                end = pos;
            }
        }
    };
    // groups of 4 consecutive bins (16-byte loads when aligned), kUnroll warp
    // steps of 32 groups per loop iteration with all loads issued first; every
    // lane of a warp runs the same number of iterations, so each match sees all
    // 32 lanes
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
        for (int u = 0; u < kUnroll; ++u) {
            if constexpr (kMode == 2) {
#pragma unroll
                for (int k = 0; k < 4; ++k) add(v[u][k]);
            } else {
                add_runs(v[u]);
            }
        }
    }
    if constexpr (kMode != 0) {
        __syncthreads();
        for (int b = threadIdx.x; b < nbins; b += blockDim.x) {
            unsigned long long c = 0;
            for (int w = 0; w < copies; ++w) c += sh[w * nbins + b];
            if (c) atomicAdd(&counts[b], c);
        }
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
    // shared histograms: a few CTAs per SM, each flush costs nbins atomics
    if (nbins <= kWarpCopyBins)
        return launch_mode<2>(bins, n, nbins, counts, grid_of(2, 4), nbins * 4 * (kHistThreads / 32), vec, s);
    if (nbins <= kSmemBins)
        return launch_mode<1>(bins, n, nbins, counts, grid_of(nbins <= 8192 ? 2 : 1, 4), nbins * 4, vec, s);
    return launch_mode<0>(bins, n, nbins, counts, grid_of(4, 4), 0, vec, s);
}

}  // namespace scg
