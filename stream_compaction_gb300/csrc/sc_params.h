// Internal launch parameters shared by the host dispatcher and the kernels.
// Not part of the public C ABI.
#pragma once
#include <cstdint>

namespace scg {

// Flag values stored in the low two bits of a look-back status word.
enum : unsigned { ST_INVALID = 0u, ST_AGGREGATE = 1u, ST_PREFIX = 2u, ST_POISON = 3u };

// Device error word values (mirrors sc_status codes of the public header).
enum : unsigned { DEV_OK = 0u, DEV_LOOKBACK_TIMEOUT = 5u, DEV_INTERNAL = 6u };

struct LookbackCtl {
    unsigned long long* status;     // one (or two) 64-bit words per tile
    unsigned long long* counter;    // dynamic tile counter (monotone across calls)
    unsigned int* error;            // device error word
    unsigned long long counter_base;
    unsigned int epoch;             // 1 .. 2^30-1; words of other epochs read as "not yet"
    unsigned int num_tiles;
    int static_ids;                 // 1: tile = blockIdx.x (the whole grid is resident at once), 0: from the counter
    long long stall_tile;           // test hook: tile that never publishes (-1: off)
    long long delay_tile;           // test hook: tile that sleeps before publishing (-1: off)
    unsigned int delay_ns;
    unsigned long long timeout_ns;  // bound on any single look-back wait
    unsigned long long* stats;      // instrumented variants only: 8 counters (see sc_scan.cuh)
    unsigned int stride_words;      // 64-bit words from one tile's status to the next (0: packed)
};

struct ScanParams {
    const void* in;
    void* out;
    long long n;                    // elements
    long long seg_len;              // > 0: independent segments of this length (batched rows)
    const unsigned char* heads;     // non-null: heads[i] != 0 starts a segment at i (seg_len unused)
    int vec_ok;                     // in and out are 16-byte aligned
    const void* carry_in;           // optional carry folded in front of element 0 (device)
    void* carry_out;                // optional inclusive total, written by the last tile (device)
    LookbackCtl lb;
};

// Canonical predicate: integers keep x when lo <= x <= hi, xor invert;
// floats keep x when (x cmp tf), with cmp in {GT, GE, LT, LE, EQ, NE},
// or always / never.
enum : int { FCMP_GT = 0, FCMP_GE, FCMP_LT, FCMP_LE, FCMP_EQ, FCMP_NE, FCMP_NEVER, FCMP_ALWAYS };

struct PredParams {
    long long lo, hi;               // integer interval (already clamped to the type)
    int invert;
    int fcmp;
    float tf;
};

struct CompactParams {
    const void* in;
    void* out;
    long long* count;               // device int64
    long long n;
    int vec_ok;
    PredParams pred;
    LookbackCtl lb;
};

struct HierParams {
    const void* in;
    void* out;
    void* totals;                   // per-tile aggregates written by the tile pass
    const void* offsets;            // per-tile exclusive offsets read by the add pass
    long long n;
    int vec_ok;
};

}  // namespace scg
