// Radix sort of uint32 keys: one stable counting-sort pass per digit.
//
// "Lecture 7: Parallel pattern -- prefix sum / scan" (UIUC ECE408 notes),
// section 2: a radix sort makes one pass per digit, a split by the digit whose
// placement is a scan; "Chapter 9 Parallel Patterns: Prefix Sum - Scan
// Algorithms" (PMPP notes), section 4.2: the scan of the digit histogram gives
// where each bucket starts.  A key with digit d in tile t goes to
//
//   (keys with a smaller digit) + (keys with digit d in tiles before t)
//     + (keys with digit d earlier in tile t).
//
// The first two terms are one exclusive scan of the tiles' digit counts laid
// out digit-major (count[d * ntiles + t]): three launches per pass,
//
//   radix_count_kernel  each tile's 256 digit counts (per-warp shared
//                       histograms);
//   the library's scan  exclusive uint32 sum over the counts, in place;
//   radix_place_kernel  each tile ranks its keys (in element order: the lanes
//                       of a warp step with the same digit, found by a match on
//                       the top digit bits and one ballot per lower bit, plus
//                       per-warp running counts per digit),
//                       reorders them by digit in shared memory and writes
//                       each digit's run at the scanned offset.
//
// Measured on GB300: a single-kernel form with a decoupled look-back per digit
// (256 chains per tile) spent its time walking those chains (about 1.4 ms per
// pass of 2^27 keys); the counts-scan-place form reads the keys twice but has
// no chains.
#include <algorithm>

#include "sc_device.cuh"
#include "sc_launch.h"

namespace scg {

namespace {

constexpr int kRadix = 256;
constexpr int kNT = 256;              // one thread per digit in the per-digit steps
constexpr int kKPT = 16;              // keys per thread
constexpr int kTileKeys = kNT * kKPT; // 4096
constexpr int kNW = kNT / 32;
constexpr int kHistNT = 512;
static_assert(kNT == kRadix, "thread d handles digit d");

// Digit counts of tile blockIdx.x into counts[d * ntiles + tile]: one shared
// histogram per warp (plain shared atomics), summed per digit.
__global__ void __launch_bounds__(kNT) radix_count_kernel(const uint32_t* __restrict__ keys, long long n, int shift,
                                                          uint32_t mask, uint32_t* __restrict__ counts,
                                                          long long ntiles) {
    __shared__ unsigned int h[kNW][kRadix];
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < kNW * kRadix; i += kNT) (&h[0][0])[i] = 0u;
    __syncthreads();
    const long long tile = blockIdx.x;
    const long long t0 = tile * kTileKeys;
    const bool full = t0 + kTileKeys <= n && (reinterpret_cast<uintptr_t>(keys) % 16) == 0;
    constexpr int kVec = kKPT / 4;
    if (full) {
        const uint4* src = reinterpret_cast<const uint4*>(keys + t0);
        uint4 q[kVec];
#pragma unroll
        for (int v = 0; v < kVec; ++v) q[v] = __ldg(src + v * kNT + tid);  // coalesced 16-byte loads
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
            atomicAdd(&h[warp][(q[v].x >> shift) & mask], 1u);
            atomicAdd(&h[warp][(q[v].y >> shift) & mask], 1u);
            atomicAdd(&h[warp][(q[v].z >> shift) & mask], 1u);
            atomicAdd(&h[warp][(q[v].w >> shift) & mask], 1u);
        }
    } else {
        for (long long i = t0 + tid; i < min(n, t0 + kTileKeys); i += kNT)
            atomicAdd(&h[warp][(__ldg(keys + i) >> shift) & mask], 1u);
    }
    __syncthreads();
    uint32_t c = 0;
#pragma unroll
    for (int w = 0; w < kNW; ++w) c += h[w][tid];
    counts[(long long)tid * ntiles + tile] = c;
}

// Block-wide exclusive scan over the 256 threads (one value each).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t x, uint32_t* scratch /* kNW entries */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    uint32_t before = 0;
#pragma unroll
    for (int w = 0; w < kNW; ++w) before += w < warp ? scratch[w] : 0u;
    return before + incl - x;
}

// Lanes of the warp whose 8-bit digit equals this lane's: __match_any_sync on
// the top kMatchBits bits, one ballot for each lower bit.  The match runs on the
// SM's address-divergence unit and its cost grows with the number of distinct
// values (about 60 cycles a call for 8 random bits, which bounded the whole
// kernel); the ballots cost integer-pipe instructions.  Splitting the bits puts
// part of the work on each.
template <int kMatchBits>
__device__ __forceinline__ uint32_t same_digit_lanes(uint32_t d) {
    uint32_t m = kMatchBits > 0 ? __match_any_sync(0xffffffffu, d >> (8 - kMatchBits)) : 0xffffffffu;
#pragma unroll
    for (int b = 0; b < 8 - kMatchBits; ++b) {
        const uint32_t bit = (d >> b) & 1u;
        const uint32_t on = __ballot_sync(0xffffffffu, bit);
        m &= on ^ (bit - 1u);                 // lanes whose bit b equals mine
    }
    return m;
}

// Load the warp's 512 keys of the tile (slot j of lane l is element
// wbase + 32 j + l) and rank each among the warp's earlier keys of its digit:
// rank = this warp's running count of the digit + same-digit lanes below.
template <bool kFull, int kMatchBits>
__device__ __forceinline__ void load_and_rank(const uint32_t* __restrict__ src, int wbase, int nvalid, int shift,
                                              uint32_t mask, uint32_t* cnt /* this warp's 256 counts */,
                                              uint32_t (&key)[kKPT], uint32_t (&rank)[kKPT]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < kKPT; ++j) {
        const int e = wbase + j * 32 + lane;
        key[j] = (kFull || e < nvalid) ? __ldg(src + j * 32) : 0u;
    }
    const uint32_t below = lanemask_lt();
#pragma unroll
    for (int j = 0; j < kKPT; ++j) {
        const bool valid = kFull || wbase + j * 32 + lane < nvalid;
        const uint32_t d = (key[j] >> shift) & mask;
        uint32_t m = same_digit_lanes<kMatchBits>(d);
        if (!kFull) m &= __ballot_sync(0xffffffffu, valid);
        const uint32_t c = cnt[d];
        rank[j] = c + __popc(m & below);
        __syncwarp();
        if (valid) cnt[d] = c + __popc(m);    // every lane of the group writes the same value
        __syncwarp();
    }
}

}  // namespace

// Place the keys of tile blockIdx.x: offsets[d * ntiles + tile] is where its
// first key with digit d goes (the scanned counts).
template <int kMatchBits>
__global__ void __launch_bounds__(kNT, 4) radix_place_kernel(const uint32_t* __restrict__ in, uint32_t* __restrict__ out,
                                                             long long n, int shift, uint32_t mask,
                                                             const uint32_t* __restrict__ offsets, long long ntiles,
                                                             unsigned int* error) {
    __shared__ uint32_t s_keys[kTileKeys];
    __shared__ __align__(16) uint32_t s_cnt[kNW][kRadix];  // running counts, then each warp's first slot per digit
    __shared__ uint32_t s_gdelta[kRadix];                   // output position of tile slot i, digit d: s_gdelta[d] + i
    __shared__ uint32_t s_scan[kNW];

    const int tid = threadIdx.x, warp = tid >> 5;
    static_assert(kNW * kRadix == 2 * 4 * kNT, "two 16-byte stores per thread clear the counts");
    reinterpret_cast<uint4*>(&s_cnt[0][0])[tid] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(&s_cnt[0][0])[tid + kNT] = make_uint4(0u, 0u, 0u, 0u);
    const long long tile = blockIdx.x;
    const long long t0 = tile * kTileKeys;
    const int nvalid = (int)min((long long)kTileKeys, n - t0);
    const uint32_t gbase = __ldg(offsets + (long long)tid * ntiles + tile);  // digit d = tid
    __syncthreads();

    uint32_t key[kKPT], rank[kKPT];
    const int wbase = warp * 32 * kKPT;
    const uint32_t* src = in + t0 + wbase + (tid & 31);
    if (nvalid == kTileKeys) load_and_rank<true, kMatchBits>(src, wbase, nvalid, shift, mask, s_cnt[warp], key, rank);
    else load_and_rank<false, kMatchBits>(src, wbase, nvalid, shift, mask, s_cnt[warp], key, rank);
    __syncthreads();

    // per digit d = tid: the tile's count, its first slot in the reordered tile,
    // and each warp's first slot
    const int d = tid;
    uint32_t tcount = 0;
#pragma unroll
    for (int w = 0; w < kNW; ++w) tcount += s_cnt[w][d];
    const uint32_t tstart = block_exclusive_scan(tcount, s_scan);
    uint32_t run = tstart;
#pragma unroll
    for (int w = 0; w < kNW; ++w) {
        const uint32_t x = s_cnt[w][d];
        s_cnt[w][d] = run;
        run += x;
    }
    s_gdelta[d] = gbase - tstart;             // mod 2^32; every position is below n < 2^32
    __syncthreads();

    // reorder the tile by digit in shared memory, then write each digit's run
#pragma unroll
    for (int j = 0; j < kKPT; ++j) {
        if (nvalid == kTileKeys || wbase + j * 32 + (tid & 31) < nvalid) {
            const uint32_t slot = s_cnt[warp][(key[j] >> shift) & mask] + rank[j];
            if (slot < (uint32_t)kTileKeys) s_keys[slot] = key[j];
            else raise_error(error, DEV_INTERNAL);  // ranks and counts disagree: never expected
        }
    }
    __syncthreads();
#pragma unroll 4
    for (int i = tid; i < nvalid; i += kNT) {
        const uint32_t k = s_keys[i];
        const uint32_t pos = s_gdelta[(k >> shift) & mask] + (uint32_t)i;
        if (pos < (uint32_t)n) out[pos] = k;  // n < 2^32
        else raise_error(error, DEV_INTERNAL);  // counts and placement disagree: never expected
    }
}

int radix_tile_keys() { return kTileKeys; }

cudaError_t launch_radix_count(const uint32_t* keys, long long n, int shift, uint32_t mask, uint32_t* counts,
                               long long ntiles, cudaStream_t s) {
    radix_count_kernel<<<(unsigned)ntiles, kNT, 0, s>>>(keys, n, shift, mask, counts, ntiles);
    return cudaGetLastError();
}

int radix_num_variants() { return 6; }

cudaError_t launch_radix_place(const uint32_t* in, uint32_t* out, long long n, int shift, uint32_t mask,
                               const uint32_t* offsets, long long ntiles, unsigned int* error, int variant,
                               cudaStream_t s) {
    auto go = [&](auto kernel) {
        kernel<<<(unsigned)ntiles, kNT, 0, s>>>(in, out, n, shift, mask, offsets, ntiles, error);
        return cudaGetLastError();
    };
    switch (variant) {  // 1 + the number of digit bits matched by __match_any_sync; 0 the default
        case 1: return go(radix_place_kernel<0>);
        case 2: return go(radix_place_kernel<1>);
        case 3: return go(radix_place_kernel<2>);
        case 0:
        case 4: return go(radix_place_kernel<3>);
        case 5: return go(radix_place_kernel<4>);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace scg
