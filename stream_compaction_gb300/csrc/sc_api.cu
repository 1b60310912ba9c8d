// C ABI of the library: argument checks, workspaces, dispatch to the kernels,
// the host-buffer pipeline and the error word.  See include/sc_scan.h for the
// contract of every entry point.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cfloat>
#include <climits>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include <cuda_runtime.h>

#include "../../include/sc_scan.h"
#include "sc_launch.h"
#include "sc_shapes.h"

namespace {

using scg::CompactParams;
using scg::HierParams;
using scg::LookbackCtl;
using scg::ScanParams;

constexpr size_t kStatusOffset = 256;       // counter at 0, error word at 8
constexpr size_t kStatsOffset = 64;         // 8 phase-timer counters of instrumented variants
constexpr int64_t kMinTile = 2048;          // smallest tile of any kernel
constexpr size_t kSlotBytes = 16;           // one look-back status slot
constexpr unsigned kMaxEpoch = (1u << 30) - 1;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;
// Public variant numbers of the uint32 sum: 0 persistent TMA kernel (shape 0),
// 1 .. N the one-tile-per-CTA shapes (shape v - 1), N + 1 the instrumented TMA
// kernel, N + 1 + c (c >= 1) the persistent kernel in shape c.
constexpr int kTmaStatsVariant = scg::kNumSumU32Variants + 1;
// Up to this many elements the default path is the one-tile-per-CTA kernel:
// measured on GB300, the persistent kernel's pipeline start-up (about 9 us)
// costs more than a short scan.  For short uint32 sums the one-tile shape
// kSmallShape: with look-back statuses in L2 lines of their own, 8192-element
// tiles of 512 threads finish n = 2^20 + 17 in 10.5 us with the L2 flushed
// (7.0 us back to back), against 12.4 (8.2) for 16384-element tiles and 11.5
// (7.4) for 4096-element ones; up to 2^22 + 17 elements that shape also beats
// the persistent kernel (16.3 against 18.6 us), at 2^23 the persistent kernel
// wins (24.8 against 25.7 us).  8-byte elements (2048-element tiles on the
// one-tile kernel) cross over near 2^20 (8 MiB): int64 sums with the L2
// flushed took 14.3 / 16.4 / 24.6 / 37.9 us at 2^19 + 3 / 2^20 + 1 / 2^21 + 8
// / 2^22 on the one-tile kernel and 14.7 / 16.4 / 20.5 / 25.4 us persistent.
constexpr int64_t kSmallScanMax = int64_t(1) << 22;   // elements of 4 bytes
constexpr int64_t kSmallScanMax8 = int64_t(1) << 20;  // elements of 8 bytes
constexpr int kSmallShape = 3;  // 8192-element tiles, 512 threads x 16 items
// Scans segmented by head flags (int32/uint32 sums): 4096-element tiles, 128-tile
// look-back windows, 8 CTAs per SM; measured on GB300 with 2^27 elements and a
// head every 1024 on average: 351 us against 377 us for shape 0.
constexpr int kHeadsShape = 8;
int max_variant() { return kTmaStatsVariant + scg::tma_num_cfgs() - 1; }
// Persistent-kernel shape of a public variant, or -1 for the one-tile-per-CTA kernel.
int tma_cfg_of(int v) {
    if (v == 0 || v == kTmaStatsVariant) return 0;
    if (v > kTmaStatsVariant && v <= max_variant()) return v - kTmaStatsVariant;
    return -1;
}

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_variant{0};
std::atomic<int> g_radix_variant{0};    // placement ranking of the radix pass (scg::launch_radix_place)
std::atomic<int> g_compact_variant{0};  // 2: one tile per CTA; the others: persistent kernel shapes
std::atomic<long long> g_stall_tile{-1};
std::atomic<long long> g_delay_tile{-1};
std::atomic<unsigned> g_delay_ns{0};
std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};
// Kernel family of the calling thread's last launch (SC_PATH_*; test hook).
thread_local int g_last_path = SC_PATH_NONE;

// ------------------------------------------------------------ workspaces
struct Workspace {
    unsigned char* base = nullptr;
    size_t bytes = 0;
    bool owned = false;
    bool dirty = true;                 // needs a zeroing memset before use
    unsigned long long counter_base = 0;
    unsigned epoch = 0;
    // bytes from here on may hold data other than status words (a radix pass's
    // digit counts, the hierarchical variant's totals), which a look-back
    // must not read as statuses: cleared up to a call's status area first
    size_t junk_from = SIZE_MAX;
};

std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t lookback_bytes(int64_t n) { return kStatusOffset + kSlotBytes * (size_t)ceil_div(std::max<int64_t>(n, 1), kMinTile); }

// Workspace of (current device, stream) with at least `need` bytes, zeroed and
// ready for the next epoch.  Caller holds g_ws_mu.
// SC_OK when `s` is not capturing into a CUDA graph: the look-back epoch and
// counter base are host state that a captured call would replay unchanged.
sc_status refuse_capture(cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return SC_ERR_CUDA;
    return cs == cudaStreamCaptureStatusNone ? SC_OK : SC_ERR_UNSUPPORTED;
}

// status_need: the end of the call's look-back status area (lookback_bytes(n));
// max_epoch: the largest epoch the call's status format holds (2^30 - 1, or
// 2^7 - 1 for one-word float-float carries): past it the workspace is cleared
// and the epochs start again.
sc_status acquire_ws(cudaStream_t s, size_t need, Workspace** out, size_t status_need = 0,
                     unsigned max_epoch = kMaxEpoch) {
    const sc_status cap = refuse_capture(s);
    if (cap != SC_OK) return cap;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SC_ERR_CUDA;
    Workspace& ws = g_ws[{dev, s}];
    if (ws.bytes < need) {
        if (ws.base && !ws.owned) return SC_ERR_WORKSPACE;
        if (ws.base) {
            cudaFree(ws.base);  // synchronises the device: no kernel still uses it
            ws.base = nullptr;
            ws.bytes = 0;
        }
        const size_t bytes = std::max(need, (size_t)(1 << 20));
        void* p = nullptr;
        if (cudaMalloc(&p, bytes) != cudaSuccess) {
            cudaGetLastError();
            return SC_ERR_WORKSPACE;
        }
        ws.base = static_cast<unsigned char*>(p);
        ws.bytes = bytes;
        ws.owned = true;
        ws.dirty = true;
    }
    if (ws.dirty || ws.epoch >= max_epoch) {
        if (cudaMemsetAsync(ws.base, 0, ws.bytes, s) != cudaSuccess) return SC_ERR_CUDA;
        ws.counter_base = 0;
        ws.epoch = 0;
        ws.dirty = false;
        ws.junk_from = SIZE_MAX;
    } else if (status_need > ws.junk_from) {
        if (cudaMemsetAsync(ws.base + ws.junk_from, 0, status_need - ws.junk_from, s) != cudaSuccess) return SC_ERR_CUDA;
        ws.junk_from = status_need;
    }
    *out = &ws;
    return SC_OK;
}

LookbackCtl make_ctl(Workspace& ws, unsigned num_tiles) {
    LookbackCtl lb;
    lb.status = reinterpret_cast<unsigned long long*>(ws.base + kStatusOffset);
    lb.counter = reinterpret_cast<unsigned long long*>(ws.base);
    lb.error = reinterpret_cast<unsigned int*>(ws.base + 8);
    lb.counter_base = ws.counter_base;
    lb.epoch = ++ws.epoch;
    lb.num_tiles = num_tiles;
    lb.static_ids = 0;
    lb.stall_tile = g_stall_tile.load();
    lb.delay_tile = g_delay_tile.load();
    lb.delay_ns = g_delay_ns.load();
    lb.timeout_ns = g_timeout_ns.load();
    lb.stats = reinterpret_cast<unsigned long long*>(ws.base + kStatsOffset);
    lb.stride_words = 0;
    return lb;
}

// Status stride of a look-back over `units` tiles or chunks in a status area
// of `area` bytes (the part of the workspace reserved for the statuses of the
// call's n, lookback_bytes(n) - kStatusOffset: other data, such as the radix
// pass's digit counts, may follow it): the widest of 128, 64, 32 and 16 bytes
// that fits.  Packed
// statuses share 128-byte L2 lines (16 four-byte carries to a line), which
// many SMs poll while others write them; measured on GB300 (uint32 sum, 2^30,
// persistent kernel) packed statuses held the scan at 0.83 of the copy peak
// and statuses in lines of their own reach 0.98.  sc_set_status_stride
// overrides the choice (g_status_stride).
std::atomic<int> g_status_stride{0};
unsigned status_stride_words(size_t area, int64_t units) {
    const int forced = g_status_stride.load();
    if (forced < 0) return 0;
    for (size_t b = 128; b >= 16; b /= 2)
        if ((forced == 0 || (size_t)forced == b) && (size_t)(units - 1) * b + 16 <= area) return (unsigned)(b / 8);
    return 0;
}

// After a launch: every CTA of the grid takes exactly one tile id, so the
// counter moved by num_tiles.  A failed launch leaves the counter unknown.
sc_status finish_launch(Workspace& ws, unsigned num_tiles, cudaError_t e) {
    g_launches.fetch_add(1);
    if (e != cudaSuccess) {
        ws.dirty = true;
        return SC_ERR_CUDA;
    }
    ws.counter_base += num_tiles;
    return SC_OK;
}

// ------------------------------------------------------------ validation
int elem_bytes(sc_dtype d) {
    switch (d) {
    case SC_I32: case SC_U32: case SC_F32: return 4;
    case SC_AFFINE_U32: case SC_I64: case SC_U64: case SC_F64: case SC_MAXCOUNT_I32: return 8;
    default: return 0;
    }
}

bool valid_dtype(int d) { return d >= SC_I32 && d <= SC_MAXCOUNT_I32; }
bool valid_op(int o) { return o >= SC_SUM && o <= SC_XOR; }

// The operator id (scg::ScanOpId) of a (dtype, op) pair; -1 unsupported.
int op_id(sc_dtype d, sc_op o) {
    using namespace scg;
    const bool i32 = d == SC_I32 || d == SC_U32, i64 = d == SC_I64 || d == SC_U64;
    switch (o) {
    case SC_SUM:
        return i32 ? OID_SUM_U32 : i64 ? OID_SUM_U64 : d == SC_F32 ? OID_SUM_F32 : d == SC_F64 ? OID_SUM_F64 : -1;
    case SC_PROD: return i32 ? OID_PROD_U32 : i64 ? OID_PROD_U64 : -1;
    case SC_AND: return i32 ? OID_AND_U32 : i64 ? OID_AND_U64 : -1;
    case SC_OR: return i32 ? OID_OR_U32 : i64 ? OID_OR_U64 : -1;
    case SC_XOR: return i32 ? OID_XOR_U32 : i64 ? OID_XOR_U64 : -1;
    case SC_MAX:
        switch (d) {
        case SC_I32: return OID_MAX_I32;
        case SC_U32: return OID_MAX_U32;
        case SC_I64: return OID_MAX_I64;
        case SC_U64: return OID_MAX_U64;
        case SC_F32: return OID_MAX_F32;
        case SC_F64: return OID_MAX_F64;
        case SC_MAXCOUNT_I32: return OID_MAXCOUNT_I32;
        default: return -1;
        }
    case SC_MIN:
        switch (d) {
        case SC_I32: return OID_MIN_I32;
        case SC_U32: return OID_MIN_U32;
        case SC_I64: return OID_MIN_I64;
        case SC_U64: return OID_MIN_U64;
        case SC_F32: return OID_MIN_F32;
        case SC_F64: return OID_MIN_F64;
        default: return -1;
        }
    case SC_COMPOSE: return d == SC_AFFINE_U32 ? OID_AFFINE_U32 : -1;
    default: return -1;
    }
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// in == out is fine; any other overlap is not.
bool bad_overlap(const void* a, const void* b, size_t bytes, bool allow_same) {
    if (a == b) return !allow_same;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bytes && y < x + bytes;
}

sc_status check_scan_args(sc_dtype dtype, sc_op op, const void* in, void* out, int64_t n, int* oid) {
    if (!valid_dtype(dtype) || !valid_op(op) || n < 0) return SC_ERR_INVALID;
    *oid = op_id(dtype, op);
    if (*oid < 0) return SC_ERR_UNSUPPORTED;
    if (n == 0) return SC_OK;
    if (!in || !out) return SC_ERR_INVALID;
    const int eb = elem_bytes(dtype);
    if (!aligned(in, eb) || !aligned(out, eb)) return SC_ERR_INVALID;
    if ((uint64_t)n > (uint64_t)INT64_MAX / 16) return SC_ERR_INVALID;
    if (bad_overlap(in, out, (size_t)n * eb, true)) return SC_ERR_INVALID;
    if (ceil_div(n, kMinTile) > (int64_t)INT_MAX) return SC_ERR_INVALID;  // grid.x limit
    return SC_OK;
}

cudaError_t dispatch_scan(int oid, const ScanParams& p, bool excl, bool seg, int variant, cudaStream_t s) {
    if (oid >= scg::kFirstExtraOid) return variant == 0 ? scg::launch_scan_extra(oid, p, excl, seg, 0, s)
                                                        : cudaErrorInvalidValue;
    switch (oid) {
    case 0: return scg::launch_scan<scg::OpSumU32>(p, excl, seg, variant, s);
    case 1: return scg::launch_scan<scg::OpSumF32>(p, excl, seg, variant, s);
    case 2: return scg::launch_scan<scg::OpMaxI32>(p, excl, seg, variant, s);
    case 3: return scg::launch_scan<scg::OpAffineU32>(p, excl, seg, variant, s);
    default: return cudaErrorInvalidValue;
    }
}

int num_sms() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int v = cache[dev].load();
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(v);
    }
    return v;
}

cudaError_t dispatch_scan_tma(int oid, const ScanParams& p, bool excl, unsigned grid, cudaStream_t s, bool stats,
                              int cfg) {
    if (oid >= scg::kFirstExtraOid) return (cfg == 0 && !stats) ? scg::launch_scan_extra(oid, p, excl, false, grid, s)
                                                                : cudaErrorInvalidValue;
    switch (oid) {
    case 0: return scg::launch_scan_tma<scg::OpSumU32>(p, excl, grid, s, stats, cfg);
    case 1: return scg::launch_scan_tma<scg::OpSumF32>(p, excl, grid, s, false, 0);
    case 2: return scg::launch_scan_tma<scg::OpMaxI32>(p, excl, grid, s, false, 0);
    case 3: return scg::launch_scan_tma<scg::OpAffineU32>(p, excl, grid, s, false, 0);
    default: return cudaErrorInvalidValue;
    }
}

// One single-pass scan launch (plain or segmented), with optional carries.
// Public variant 0 is the persistent TMA kernel where it applies (16-byte
// aligned, unsegmented, more than kSmallScanMax elements of 4 bytes or
// kSmallScanMax8 of 8 bytes); every other case,
// and public variants v >= 1 of the uint32 sum, use the one-tile-per-CTA
// kernel (shape v - 1; by default shape 0, kSmallShape for short uint32 sums
// and kHeadsShape for uint32 sums segmented by head flags).  Segmented scans
// and batched rows take shape v - 1 only where it has a segmented form.
sc_status run_scan(int oid, const void* in, void* out, int64_t n, int64_t seg_len, bool excl,
                   const void* carry_in, void* carry_out, cudaStream_t s, const unsigned char* heads = nullptr) {
    const bool segmented = seg_len > 0 || heads != nullptr;
    const int api_variant = oid == 0 ? g_variant.load() : 0;
    const bool vec_ok = aligned(in, 16) && aligned(out, 16);
    const int eb = scg::oid_elem_bytes(oid);
    const int cfg = tma_cfg_of(api_variant);
    scg::TmaShape sh{0, 0, 0, 0, 1, 2};
    if (cfg >= 0) scg::tma_shape(cfg, &sh);
    const int64_t tma_tile = cfg >= 0 ? sh.tile_bytes / eb : 0;
    const bool tma_stats = api_variant == kTmaStatsVariant;
    const bool small = api_variant == 0 && n <= (eb == 4 ? kSmallScanMax : kSmallScanMax8);
    const bool use_tma = cfg >= 0 && !small && !segmented && vec_ok && n >= tma_tile &&
                         n / tma_tile * (sh.tile_bytes / 128) < (int64_t)INT_MAX && num_sms() > 0;
    int legacy_variant = (small && oid == 0 && !segmented) ? kSmallShape
                         : (cfg >= 0 || api_variant == 0) ? 0 : api_variant - 1;
    if (segmented && !scg::segmented_shape(legacy_variant)) legacy_variant = 0;
    if (heads && oid == 0 && api_variant == 0) legacy_variant = kHeadsShape;
    // units of the look-back: chunks of the persistent kernel, tiles otherwise
    const int64_t tile = use_tma ? tma_tile * sh.chunk_tiles : scg::scan_tile_elems(oid, legacy_variant);
    const unsigned ntiles = (unsigned)ceil_div(n, tile);
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace* ws = nullptr;
    // float32 sums carry float-float pairs in one-word statuses with a 7-bit epoch
    const unsigned max_epoch = oid == scg::OID_SUM_F32 ? (1u << scg::kFloat2EpochBits) - 1 : kMaxEpoch;
    sc_status st = acquire_ws(s, lookback_bytes(n), &ws, lookback_bytes(n), max_epoch);
    if (st != SC_OK) return st;
    ScanParams p;
    p.in = in;
    p.out = out;
    p.n = n;
    p.seg_len = seg_len;
    p.heads = heads;
    p.vec_ok = vec_ok;
    p.carry_in = carry_in;
    p.carry_out = carry_out;
    // Batched rows of at most 8192 elements: the persistent rows kernel (no
    // look-back, one read of each element).  Rows dividing its 8192-element
    // tile: every tile holds whole rows.  Other lengths: each CTA carries the
    // fold of the open row from one tile to the next and reads back, once, the
    // part of its first tile's row before it, so those need out != in.
    const int64_t rows_tile = scg::rows_tma_tile_elems();
    if (seg_len > 0 && seg_len <= rows_tile && !heads && (rows_tile % seg_len == 0 || in != out) &&
        api_variant == 0 && scg::rows_tma_supported(oid) &&
        vec_ok && n >= rows_tile && !carry_in && !carry_out && n / rows_tile * 256 < (int64_t)INT_MAX &&
        num_sms() > 0) {
        const int64_t tiles = ceil_div(n, rows_tile);
        p.lb = make_ctl(*ws, (unsigned)tiles);
        const unsigned grid = (unsigned)std::min<int64_t>(num_sms(), tiles);
        g_last_path = SC_PATH_ROWS_PERSISTENT;
        return finish_launch(*ws, 0, scg::launch_rows_tma(oid, p, excl, grid, s));
    }
    // Other batched rows whose length divides the one-tile kernel's tile stay
    // there (every tile starts a row: no look-back at all; measured on GB300
    // with 2^28 int32, rows of 16-4096: 0.77-0.80 of the copy peak against 0.70
    // on the persistent segmented kernel); other row lengths (33, 1000, 2047:
    // 0.56 there) take the persistent segmented kernel (0.75).
    const int64_t seg_tile = scg::segscan_tma_tile_elems();
    // scans segmented by head flags, and batched rows (heads at the multiples
    // of the row length): the persistent kernel when the operator has that
    // form and the arrays are 16-byte aligned and hold a full tile
    const bool rows_fit_tiles = seg_len > 0 && scg::scan_tile_elems(oid, legacy_variant) % seg_len == 0;
    if (segmented && !rows_fit_tiles && api_variant == 0 && scg::segscan_tma_supported(oid) && vec_ok &&
        (!heads || aligned(heads, 16)) && n >= seg_tile && !carry_in && !carry_out &&
        n / seg_tile * 256 < (int64_t)INT_MAX && num_sms() > 0) {
        const unsigned nchunks = (unsigned)ceil_div(n, seg_tile * scg::segscan_tma_chunk_tiles());
        p.lb = make_ctl(*ws, nchunks);
        p.lb.stride_words = status_stride_words(lookback_bytes(n) - kStatusOffset, nchunks);
        const unsigned grid = (unsigned)std::min<int64_t>(num_sms(), nchunks);
        g_last_path = SC_PATH_SEGSCAN_PERSISTENT;
        const cudaError_t e = scg::launch_segscan_tma(oid, p, excl, grid, s);
        return finish_launch(*ws, nchunks + grid * (unsigned)scg::tma_ids_per_cta(), e);
    }
    p.lb = make_ctl(*ws, ntiles);
    if (use_tma) {
        p.lb.stride_words = status_stride_words(lookback_bytes(n) - kStatusOffset, ntiles);
        const unsigned grid = (unsigned)std::min<int64_t>((int64_t)num_sms() * sh.ctas_per_sm, ntiles);
        g_last_path = SC_PATH_SCAN_PERSISTENT;
        const cudaError_t e = dispatch_scan_tma(oid, p, excl, grid, s, tma_stats, cfg);
        return finish_launch(*ws, ntiles + grid * (unsigned)sh.ids_per_cta, e);
    }
    g_last_path = SC_PATH_SCAN_ONE_TILE;
    // a grid no larger than the SM count is resident at once, so tiles may take
    // their ids from blockIdx.x (no counter round trip): every tile a look-back
    // waits on is already running
    const int sms = num_sms();
    p.lb.static_ids = sms > 0 && ntiles <= (unsigned)sms;
    p.lb.stride_words = status_stride_words(lookback_bytes(n) - kStatusOffset, ntiles);
    return finish_launch(*ws, p.lb.static_ids ? 0u : ntiles,
                         dispatch_scan(oid, p, excl, segmented, legacy_variant, s));
}

// ------------------------------------------------------ compaction predicate
// Canonical integer form: keep x when lo <= x <= hi (xor invert), computed
// exactly from "x <pred> t" with t a double, then clamped to [tmin, tmax].
scg::PredParams int_pred(sc_pred pred, double t, double tmin, double tmax) {
    scg::PredParams q{};
    q.invert = 0;
    double lo = tmin, hi = tmax;
    bool empty = false;
    if (std::isnan(t)) {
        empty = (pred != SC_NE);  // every comparison with NaN is false, except !=
    } else {
        switch (pred) {
        case SC_GT: lo = std::floor(t) + 1.0; break;
        case SC_GE: lo = std::ceil(t); break;
        case SC_LT: hi = std::ceil(t) - 1.0; break;
        case SC_LE: hi = std::floor(t); break;
        case SC_EQ:
        case SC_NE:
            if (std::floor(t) == t) { lo = hi = t; } else { empty = true; }
            if (pred == SC_NE) q.invert = 1;
            break;
        }
    }
    lo = std::max(lo, tmin);
    hi = std::min(hi, tmax);
    if (empty || lo > hi) {
        // empty set; with invert it becomes "everything"
        q.lo = 1;
        q.hi = 0;
        if (tmin < 0) { q.lo = (long long)tmax; q.hi = (long long)tmin; }
    } else {
        q.lo = (long long)lo;
        q.hi = (long long)hi;
    }
    return q;
}

float round_down_f(double t) {
    float f = (float)t;
    if ((double)f > t) f = std::nextafter(f, -INFINITY);
    return f;
}
float round_up_f(double t) {
    float f = (float)t;
    if ((double)f < t) f = std::nextafter(f, INFINITY);
    return f;
}

// Canonical float form: an outcome mask over {x > tf, x == tf, x < tf, NaN}
// with tf chosen so that the float comparison equals the double one.
scg::PredParams float_pred(sc_pred pred, double t) {
    enum : long long { G = 1, E = 2, L = 4, U = 8 };
    scg::PredParams q{};
    q.tf = 0.0f;
    if (std::isnan(t)) {
        q.lo = (pred == SC_NE) ? (G | E | L | U) : 0;
        return q;
    }
    switch (pred) {
    case SC_GT: q.tf = round_down_f(t); q.lo = G; break;
    case SC_GE: q.tf = round_up_f(t); q.lo = G | E; break;
    case SC_LT: q.tf = round_up_f(t); q.lo = L; break;
    case SC_LE: q.tf = round_down_f(t); q.lo = L | E; break;
    case SC_EQ:
    case SC_NE: {
        const float f = (float)t;
        const bool exact = (double)f == t;
        q.tf = f;
        if (pred == SC_EQ) q.lo = exact ? E : 0;
        else q.lo = exact ? (G | L | U) : (G | E | L | U);
        break;
    }
    }
    return q;
}

// ------------------------------------------------------ host-buffer pipeline
struct HostPipe {
    static constexpr int kBufs = 3;
    bool ready = false;
    size_t buf_bytes = 0;
    void* dbuf[kBufs] = {};
    void* carry = nullptr;  // two 16-byte slots
    cudaStream_t h2d = nullptr, cmp = nullptr, d2h = nullptr;
    cudaEvent_t ev_h2d[kBufs], ev_cmp[kBufs], ev_d2h[kBufs], ev_start;
    std::mutex mu;
};
std::mutex g_pipe_mu;
std::map<std::pair<int, cudaStream_t>, HostPipe*> g_pipes;  // per (device, caller stream)
constexpr size_t kPipeBufBytes = 64ull << 20;  // 64 MiB per staging buffer

sc_status pipe_init(HostPipe& hp) {
    if (hp.ready) return SC_OK;
    for (int i = 0; i < HostPipe::kBufs; ++i)
        if (cudaMalloc(&hp.dbuf[i], kPipeBufBytes) != cudaSuccess) return SC_ERR_WORKSPACE;
    if (cudaMalloc(&hp.carry, 64) != cudaSuccess) return SC_ERR_WORKSPACE;
    if (cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.cmp, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) != cudaSuccess)
        return SC_ERR_CUDA;
    for (int i = 0; i < HostPipe::kBufs; ++i) {
        if (cudaEventCreateWithFlags(&hp.ev_h2d[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.ev_cmp[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.ev_d2h[i], cudaEventDisableTiming) != cudaSuccess)
            return SC_ERR_CUDA;
    }
    if (cudaEventCreateWithFlags(&hp.ev_start, cudaEventDisableTiming) != cudaSuccess) return SC_ERR_CUDA;
    hp.buf_bytes = kPipeBufBytes;
    hp.ready = true;
    return SC_OK;
}

// Wait for a pipe's streams, then free its staging buffers, streams and events
// (and the look-back workspace of its internal kernel stream).
sc_status pipe_destroy(HostPipe& hp, int dev) {
    sc_status st = SC_OK;
    for (cudaStream_t q : {hp.h2d, hp.cmp, hp.d2h})
        if (q && cudaStreamSynchronize(q) != cudaSuccess) st = SC_ERR_CUDA;
    for (int i = 0; i < HostPipe::kBufs; ++i)
        if (hp.dbuf[i]) cudaFree(hp.dbuf[i]);
    if (hp.carry) cudaFree(hp.carry);
    if (hp.cmp) {
        std::lock_guard<std::mutex> lk(g_ws_mu);
        auto it = g_ws.find({dev, hp.cmp});
        if (it != g_ws.end()) {
            if (it->second.owned && it->second.base) cudaFree(it->second.base);
            g_ws.erase(it);
        }
    }
    if (hp.ready) {
        for (int i = 0; i < HostPipe::kBufs; ++i) {
            cudaEventDestroy(hp.ev_h2d[i]);
            cudaEventDestroy(hp.ev_cmp[i]);
            cudaEventDestroy(hp.ev_d2h[i]);
        }
        cudaEventDestroy(hp.ev_start);
    }
    for (cudaStream_t q : {hp.h2d, hp.cmp, hp.d2h})
        if (q) cudaStreamDestroy(q);
    return st;
}

}  // namespace

// ============================================================ public ABI
extern "C" {

const char* sc_version(void) { return "sc_gb300 1.0 (sm_103a)"; }

const char* sc_status_string(sc_status s) {
    switch (s) {
    case SC_OK: return "SC_OK";
    case SC_ERR_INVALID: return "SC_ERR_INVALID: invalid argument";
    case SC_ERR_UNSUPPORTED: return "SC_ERR_UNSUPPORTED: dtype/op combination not provided";
    case SC_ERR_WORKSPACE: return "SC_ERR_WORKSPACE: workspace too small or allocation failed";
    case SC_ERR_CUDA: return "SC_ERR_CUDA: CUDA runtime error";
    case SC_ERR_LOOKBACK_TIMEOUT: return "SC_ERR_LOOKBACK_TIMEOUT: a tile gave up waiting on its predecessors";
    case SC_ERR_INTERNAL: return "SC_ERR_INTERNAL: a kernel's bounds check caught an out-of-range position";
    default: return "unknown sc_status";
    }
}

size_t sc_workspace_bytes(int64_t n) { return lookback_bytes(n < 0 ? 0 : n); }

sc_status sc_set_workspace(void* d_ws, size_t bytes, sc_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SC_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    auto it = g_ws.find({dev, s});
    if (it != g_ws.end()) {
        if (it->second.owned && it->second.base) cudaFree(it->second.base);
        g_ws.erase(it);
    }
    if (!d_ws) return SC_OK;
    if (!aligned(d_ws, 256) || bytes < lookback_bytes(1)) return SC_ERR_INVALID;
    Workspace& ws = g_ws[{dev, s}];
    ws.base = static_cast<unsigned char*>(d_ws);
    ws.bytes = bytes;
    ws.owned = false;
    ws.dirty = true;
    return SC_OK;
}

static sc_status scan_common(sc_dtype dtype, sc_op op, const void* in, void* out, int64_t n, sc_stream_t stream,
                             bool excl) {
    int oid = -1;
    sc_status st = check_scan_args(dtype, op, in, out, n, &oid);
    if (st != SC_OK || n == 0) return st;
    return run_scan(oid, in, out, n, 0, excl, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

sc_status sc_scan_inclusive(sc_dtype dtype, sc_op op, const void* in, void* out, int64_t n, sc_stream_t stream) {
    return scan_common(dtype, op, in, out, n, stream, false);
}

sc_status sc_scan_exclusive(sc_dtype dtype, sc_op op, const void* in, void* out, int64_t n, sc_stream_t stream) {
    return scan_common(dtype, op, in, out, n, stream, true);
}

// ---------------------------------------------------- histogram, bin offsets
static sc_status check_hist_args(const int32_t* bins, int64_t n, int64_t nbins, const int64_t* out, int64_t out_len) {
    if (n < 0 || nbins < 1 || nbins > (int64_t)INT32_MAX - 1) return SC_ERR_INVALID;
    if (!out || !aligned(out, 8)) return SC_ERR_INVALID;
    if (n == 0) return SC_OK;
    if (!bins || !aligned(bins, 4)) return SC_ERR_INVALID;
    const uintptr_t b = reinterpret_cast<uintptr_t>(bins), o = reinterpret_cast<uintptr_t>(out);
    if (b < o + (size_t)out_len * 8 && o < b + (size_t)n * 4) return SC_ERR_INVALID;  // the output must not overlap the bins
    return SC_OK;
}

// counts[0..zero_len) = 0, then counts[b] += occurrences of b in bins, 0 <= b < nbins.
static sc_status count_bins(const int32_t* bins, int64_t n, int64_t nbins, int64_t* counts, int64_t zero_len,
                            cudaStream_t s) {
    if (cudaMemsetAsync(counts, 0, (size_t)zero_len * 8, s) != cudaSuccess) return SC_ERR_CUDA;
    if (n == 0) return SC_OK;
    const int sms = num_sms();
    if (sms <= 0) return SC_ERR_CUDA;
    const cudaError_t e =
        scg::launch_histogram(bins, n, (int)nbins, reinterpret_cast<unsigned long long*>(counts), sms, s);
    g_launches.fetch_add(1);
    return e == cudaSuccess ? SC_OK : SC_ERR_CUDA;
}

sc_status sc_histogram(const int32_t* d_bins, int64_t n, int64_t nbins, int64_t* d_counts, sc_stream_t stream) {
    const sc_status st = check_hist_args(d_bins, n, nbins, d_counts, nbins);
    if (st != SC_OK) return st;
    return count_bins(d_bins, n, nbins, d_counts, nbins, reinterpret_cast<cudaStream_t>(stream));
}

sc_status sc_bin_offsets(const int32_t* d_bins, int64_t n, int64_t nbins, int64_t* d_offsets, sc_stream_t stream) {
    const sc_status st = check_hist_args(d_bins, n, nbins, d_offsets, nbins + 1);
    if (st != SC_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n > 0 || nbins > 0) {
        const sc_status cap = refuse_capture(s);  // before the first launch
        if (cap != SC_OK) return cap;
    }
    // counts in offsets[0..nbins), 0 in offsets[nbins]; the exclusive scan in
    // place then leaves the total in offsets[nbins]
    const sc_status r = count_bins(d_bins, n, nbins, d_offsets, nbins + 1, s);
    if (r != SC_OK) return r;
    return run_scan(scg::OID_SUM_U64, d_offsets, d_offsets, nbins + 1, 0, true, nullptr, nullptr, s);
}

// ------------------------------------------------------------- radix sort
static bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bbytes && y < x + abytes;
}

// One pass: counts of each tile's digits (digit-major), their exclusive scan in
// place (bucket start + the earlier tiles' keys of the digit, in one value),
// then the placement.  The counts live in the stream's workspace after the
// scan's own status words.
static sc_status radix_one_pass(const uint32_t* in, uint32_t* out, int64_t n, int shift, uint32_t mask,
                                cudaStream_t s) {
    const int64_t ntiles = ceil_div(n, scg::radix_tile_keys());
    const int64_t m = 256 * ntiles;
    const size_t counts_off = (lookback_bytes(m) + 255) / 256 * 256;
    unsigned char* base = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_ws_mu);
        Workspace* ws = nullptr;
        const sc_status st = acquire_ws(s, counts_off + (size_t)m * 4, &ws, lookback_bytes(m));
        if (st != SC_OK) return st;
        base = ws->base;
        ws->junk_from = std::min(ws->junk_from, counts_off);  // the digit counts follow the scan's statuses
    }
    uint32_t* counts = reinterpret_cast<uint32_t*>(base + counts_off);
    cudaError_t e = scg::launch_radix_count(in, n, shift, mask, counts, ntiles, s);
    g_launches.fetch_add(1);
    if (e != cudaSuccess) return SC_ERR_CUDA;
    // the scan needs fewer workspace bytes than acquired above: no reallocation
    sc_status st = run_scan(scg::OID_SUM_U32, counts, counts, m, 0, true, nullptr, nullptr, s);
    if (st != SC_OK) return st;
    e = scg::launch_radix_place(in, out, n, shift, mask, counts, ntiles, reinterpret_cast<unsigned int*>(base + 8),
                                g_radix_variant.load(), s);
    g_launches.fetch_add(1);
    return e == cudaSuccess ? SC_OK : SC_ERR_CUDA;
}

sc_status sc_radix_pass_u32(const uint32_t* d_in, uint32_t* d_out, int64_t n, int shift, int bits,
                            sc_stream_t stream) {
    if (n < 0 || n > (int64_t)UINT32_MAX || bits < 1 || bits > 8 || shift < 0 || shift > 31) return SC_ERR_INVALID;
    if (n == 0) return SC_OK;
    if (!d_in || !d_out || !aligned(d_in, 4) || !aligned(d_out, 4)) return SC_ERR_INVALID;
    if (overlaps(d_in, (size_t)n * 4, d_out, (size_t)n * 4)) return SC_ERR_INVALID;
    return radix_one_pass(d_in, d_out, n, shift, (1u << bits) - 1u, reinterpret_cast<cudaStream_t>(stream));
}

sc_status sc_radix_sort_u32(const uint32_t* d_in, uint32_t* d_out, uint32_t* d_tmp, int64_t n, sc_stream_t stream) {
    if (n < 0 || n > (int64_t)UINT32_MAX) return SC_ERR_INVALID;
    if (n == 0) return SC_OK;
    if (!d_in || !d_out || !d_tmp || !aligned(d_in, 4) || !aligned(d_out, 4) || !aligned(d_tmp, 4))
        return SC_ERR_INVALID;
    const size_t bytes = (size_t)n * 4;
    if (overlaps(d_tmp, bytes, d_in, bytes) || overlaps(d_tmp, bytes, d_out, bytes)) return SC_ERR_INVALID;
    if (d_in != d_out && overlaps(d_in, bytes, d_out, bytes)) return SC_ERR_INVALID;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // least significant digit first: in -> tmp -> out -> tmp -> out
    const uint32_t* src[4] = {d_in, d_tmp, d_out, d_tmp};
    uint32_t* dst[4] = {d_tmp, d_out, d_tmp, d_out};
    for (int k = 0; k < 4; ++k) {
        const sc_status st = radix_one_pass(src[k], dst[k], n, 8 * k, 0xffu, s);
        if (st != SC_OK) return st;
    }
    return SC_OK;
}

sc_status sc_scan_segmented(sc_dtype dtype, sc_op op, int exclusive, const void* in, const uint8_t* d_heads,
                            void* out, int64_t n, sc_stream_t stream) {
    int oid = -1;
    sc_status st = check_scan_args(dtype, op, in, out, n, &oid);
    if (st != SC_OK || n == 0) return st;
    if (!d_heads) return SC_ERR_INVALID;
    const uintptr_t h = reinterpret_cast<uintptr_t>(d_heads), o = reinterpret_cast<uintptr_t>(out);
    const size_t out_bytes = (size_t)n * elem_bytes(dtype);
    if (h < o + out_bytes && o < h + (size_t)n) return SC_ERR_INVALID;  // the flags must not be overwritten
    return run_scan(oid, in, out, n, 0, exclusive != 0, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream),
                    d_heads);
}

sc_status sc_scan_batched(sc_dtype dtype, sc_op op, int exclusive, const void* in, void* out, int64_t rows,
                          int64_t cols, sc_stream_t stream) {
    if (rows < 0 || cols < 0) return SC_ERR_INVALID;
    if (cols > 0 && rows > INT64_MAX / cols) return SC_ERR_INVALID;
    const int64_t n = rows * cols;
    int oid = -1;
    sc_status st = check_scan_args(dtype, op, in, out, n, &oid);
    if (st != SC_OK || n == 0) return st;
    const int64_t seg = rows == 1 ? 0 : cols;
    return run_scan(oid, in, out, n, seg, exclusive != 0, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

sc_status sc_compact_if(sc_dtype dtype, const void* in, void* out, int64_t* d_count, int64_t n, sc_pred pred,
                        double threshold, sc_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!valid_dtype(dtype) || n < 0 || pred < SC_GT || pred > SC_NE) return SC_ERR_INVALID;
    if (dtype != SC_I32 && dtype != SC_U32 && dtype != SC_F32) return SC_ERR_UNSUPPORTED;
    if (!d_count || !aligned(d_count, 8)) return SC_ERR_INVALID;
    if (n == 0) {
        if (cudaMemsetAsync(d_count, 0, sizeof(int64_t), s) != cudaSuccess) return SC_ERR_CUDA;
        return SC_OK;
    }
    if (!in || !out || !aligned(in, 4) || !aligned(out, 4)) return SC_ERR_INVALID;
    if ((uint64_t)n > (uint64_t)INT64_MAX / 16) return SC_ERR_INVALID;
    if (bad_overlap(in, out, (size_t)n * 4, false)) return SC_ERR_INVALID;
    if (ceil_div(n, scg::CompactConfig::TILE) > (int64_t)INT_MAX) return SC_ERR_INVALID;

    CompactParams p;
    p.in = in;
    p.out = out;
    p.count = reinterpret_cast<long long*>(d_count);
    p.n = n;
    p.vec_ok = aligned(in, 16);
    if (dtype == SC_I32) p.pred = int_pred(pred, threshold, (double)INT32_MIN, (double)INT32_MAX);
    else if (dtype == SC_U32) p.pred = int_pred(pred, threshold, 0.0, (double)UINT32_MAX);
    else p.pred = float_pred(pred, threshold);

    const bool wide = n > (int64_t)UINT32_MAX;
    // persistent kernel for 16-byte aligned inputs of at least one full tile
    const int64_t ptile = scg::compact_tma_tile_elems();
    const int cvar = g_compact_variant.load();
    const bool use_tma = p.vec_ok && n >= ptile && n / ptile * (ptile * 4 / 128) < (int64_t)INT_MAX && num_sms() > 0 &&
                         cvar != 2;
    // public variant -> persistent kernel shape (3: packed stores, 4: 4 + 2 stages, 5: 2 + 4 stages,
    // 6 and 7: lag 6 and 4)
    const int tma_shape_id = cvar >= 3 ? cvar - 1 : cvar;
    const int64_t unit = use_tma ? ptile * scg::compact_tma_chunk_tiles() : scg::CompactConfig::TILE;
    const unsigned ntiles = (unsigned)ceil_div(n, unit);
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace* ws = nullptr;
    sc_status st = acquire_ws(s, lookback_bytes(n), &ws, lookback_bytes(n));
    if (st != SC_OK) return st;
    p.lb = make_ctl(*ws, ntiles);
    p.lb.stride_words = status_stride_words(lookback_bytes(n) - kStatusOffset, ntiles);
    cudaError_t e;
    if (use_tma) {
        const unsigned grid = (unsigned)std::min<int64_t>(num_sms(), ntiles);
        if (dtype == SC_I32) e = scg::launch_compact_tma<int32_t>(p, wide, grid, s, tma_shape_id);
        else if (dtype == SC_U32) e = scg::launch_compact_tma<uint32_t>(p, wide, grid, s, tma_shape_id);
        else e = scg::launch_compact_tma<float>(p, wide, grid, s, tma_shape_id);
        g_last_path = SC_PATH_COMPACT_PERSISTENT;
        return finish_launch(*ws, ntiles + grid * (unsigned)scg::tma_ids_per_cta(), e);
    }
    g_last_path = SC_PATH_COMPACT_ONE_TILE;
    if (dtype == SC_I32) e = scg::launch_compact<int32_t>(p, wide, s);
    else if (dtype == SC_U32) e = scg::launch_compact<uint32_t>(p, wide, s);
    else e = scg::launch_compact<float>(p, wide, s);
    return finish_launch(*ws, ntiles, e);
}

size_t sc_hier_workspace_bytes(sc_dtype dtype, int64_t n) {
    if (!valid_dtype(dtype) || n <= 0) return 0;
    if (dtype != SC_I32 && dtype != SC_U32 && dtype != SC_F32 && dtype != SC_AFFINE_U32) return 0;
    const int oid = dtype == SC_AFFINE_U32 ? 3 : 0;
    const int64_t t = scg::hier_tile_elems(oid);
    size_t total = 0;
    for (int64_t m = n; m > 1;) {
        const int64_t k = ceil_div(m, t);
        total += (size_t)ceil_div(k * elem_bytes(dtype), 256) * 256;
        m = k;
    }
    return total + 256;
}

static cudaError_t dispatch_hier_tiles(int oid, const HierParams& p, bool excl, unsigned nt, cudaStream_t s) {
    switch (oid) {
    case 0: return scg::launch_hier_tiles<scg::OpSumU32>(p, excl, nt, s);
    case 1: return scg::launch_hier_tiles<scg::OpSumF32>(p, excl, nt, s);
    case 2: return scg::launch_hier_tiles<scg::OpMaxI32>(p, excl, nt, s);
    case 3: return scg::launch_hier_tiles<scg::OpAffineU32>(p, excl, nt, s);
    default: return cudaErrorInvalidValue;
    }
}
static cudaError_t dispatch_hier_add(int oid, const HierParams& p, unsigned nt, cudaStream_t s) {
    switch (oid) {
    case 0: return scg::launch_hier_add<scg::OpSumU32>(p, nt, s);
    case 1: return scg::launch_hier_add<scg::OpSumF32>(p, nt, s);
    case 2: return scg::launch_hier_add<scg::OpMaxI32>(p, nt, s);
    case 3: return scg::launch_hier_add<scg::OpAffineU32>(p, nt, s);
    default: return cudaErrorInvalidValue;
    }
}

// Level l: scan `in` (m elements) into `out` tile by tile, totals into
// level_buf[l]; recursively exclusive-scan the totals in place; add them back.
static sc_status hier_level(int oid, int eb, const void* in, void* out, int64_t m, bool excl, unsigned char* scratch,
                            size_t scratch_off, cudaStream_t s) {
    const int64_t t = scg::hier_tile_elems(oid);
    const unsigned nt = (unsigned)ceil_div(m, t);
    void* totals = scratch + scratch_off;
    const size_t next_off = scratch_off + (size_t)ceil_div((int64_t)nt * eb, 256) * 256;
    HierParams p;
    p.in = in;
    p.out = out;
    p.totals = totals;
    p.offsets = totals;
    p.n = m;
    p.vec_ok = aligned(in, 16) && aligned(out, 16);
    cudaError_t e = dispatch_hier_tiles(oid, p, excl, nt, s);
    g_launches.fetch_add(1);
    if (e != cudaSuccess) return SC_ERR_CUDA;
    if (nt > 1) {
        sc_status st = hier_level(oid, eb, totals, totals, nt, true, scratch, next_off, s);
        if (st != SC_OK) return st;
        e = dispatch_hier_add(oid, p, nt, s);
        g_launches.fetch_add(1);
        if (e != cudaSuccess) return SC_ERR_CUDA;
    }
    return SC_OK;
}

sc_status sc_scan_hierarchical(sc_dtype dtype, sc_op op, int exclusive, const void* in, void* out, int64_t n,
                               sc_stream_t stream) {
    int oid = -1;
    sc_status st = check_scan_args(dtype, op, in, out, n, &oid);
    if (st != SC_OK) return st;
    if (oid >= scg::kFirstExtraOid) return SC_ERR_UNSUPPORTED;
    if (n == 0) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t need = kStatusOffset + sc_hier_workspace_bytes(dtype, n);
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace* ws = nullptr;
    st = acquire_ws(s, std::max(need, lookback_bytes(n)), &ws);
    if (st != SC_OK) return st;
    ws->junk_from = kStatusOffset;  // per-level totals where statuses go
    return hier_level(oid, elem_bytes(dtype), in, out, n, exclusive != 0, ws->base, kStatusOffset, s);
}

sc_status sc_scan_host(sc_dtype dtype, sc_op op, int exclusive, const void* h_in, void* h_out, int64_t n,
                       sc_stream_t stream) {
    int oid = -1;
    if (!valid_dtype(dtype) || !valid_op(op) || n < 0) return SC_ERR_INVALID;
    oid = op_id(dtype, op);
    if (oid < 0) return SC_ERR_UNSUPPORTED;
    if (n == 0) return SC_OK;
    if (!h_in || !h_out) return SC_ERR_INVALID;
    const int eb = elem_bytes(dtype);
    if (bad_overlap(h_in, h_out, (size_t)n * eb, true)) return SC_ERR_INVALID;
    const sc_status cap = refuse_capture(reinterpret_cast<cudaStream_t>(stream));
    if (cap != SC_OK) return cap;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SC_ERR_CUDA;
    HostPipe* hp;
    {
        std::lock_guard<std::mutex> lk(g_pipe_mu);
        HostPipe*& slot = g_pipes[{dev, reinterpret_cast<cudaStream_t>(stream)}];
        if (!slot) slot = new HostPipe();
        hp = slot;
    }
    std::lock_guard<std::mutex> lk(hp->mu);
    sc_status st = pipe_init(*hp);
    if (st != SC_OK) return st;
    cudaStream_t caller = reinterpret_cast<cudaStream_t>(stream);
    const int64_t chunk = (int64_t)(hp->buf_bytes / eb);
    const int64_t nchunks = ceil_div(n, chunk);
    if (cudaEventRecord(hp->ev_start, caller) != cudaSuccess) return SC_ERR_CUDA;
    cudaStreamWaitEvent(hp->h2d, hp->ev_start, 0);
    cudaStreamWaitEvent(hp->cmp, hp->ev_start, 0);
    const unsigned char* src = static_cast<const unsigned char*>(h_in);
    unsigned char* dst = static_cast<unsigned char*>(h_out);
    unsigned char* carry = static_cast<unsigned char*>(hp->carry);
    for (int64_t i = 0; i < nchunks; ++i) {
        const int b = (int)(i % HostPipe::kBufs);
        const int64_t off = i * chunk;
        const int64_t cn = std::min(chunk, n - off);
        const size_t bytes = (size_t)cn * eb;
        if (i >= HostPipe::kBufs) cudaStreamWaitEvent(hp->h2d, hp->ev_d2h[b], 0);
        if (cudaMemcpyAsync(hp->dbuf[b], src + off * eb, bytes, cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess)
            return SC_ERR_CUDA;
        cudaEventRecord(hp->ev_h2d[b], hp->h2d);
        cudaStreamWaitEvent(hp->cmp, hp->ev_h2d[b], 0);
        const void* cin = i > 0 ? carry + 16 * ((i - 1) & 1) : nullptr;
        void* cout = carry + 16 * (i & 1);
        st = run_scan(oid, hp->dbuf[b], hp->dbuf[b], cn, 0, exclusive != 0, cin, cout, hp->cmp);
        if (st != SC_OK) return st;
        cudaEventRecord(hp->ev_cmp[b], hp->cmp);
        cudaStreamWaitEvent(hp->d2h, hp->ev_cmp[b], 0);
        if (cudaMemcpyAsync(dst + off * eb, hp->dbuf[b], bytes, cudaMemcpyDeviceToHost, hp->d2h) != cudaSuccess)
            return SC_ERR_CUDA;
        cudaEventRecord(hp->ev_d2h[b], hp->d2h);
    }
    if (cudaStreamSynchronize(hp->d2h) != cudaSuccess || cudaStreamSynchronize(hp->cmp) != cudaSuccess)
        return SC_ERR_CUDA;
    return sc_get_device_error(reinterpret_cast<sc_stream_t>(hp->cmp));
}

sc_status sc_get_device_error(sc_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SC_ERR_CUDA;
    unsigned int* err = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_ws_mu);
        auto it = g_ws.find({dev, s});
        if (it != g_ws.end() && it->second.base) err = reinterpret_cast<unsigned int*>(it->second.base + 8);
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return SC_ERR_CUDA;
    if (!err) return SC_OK;
    unsigned int h = 0;
    if (cudaMemcpy(&h, err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return SC_ERR_CUDA;
    if (h != 0) {
        if (cudaMemset(err, 0, sizeof(h)) != cudaSuccess) return SC_ERR_CUDA;
        // a kernel that gave up may not have consumed its tile ids: start the
        // next call from a cleared workspace
        std::lock_guard<std::mutex> lk(g_ws_mu);
        auto it = g_ws.find({dev, s});
        if (it != g_ws.end()) it->second.dirty = true;
        return (sc_status)h;
    }
    return SC_OK;
}

uint64_t sc_launch_count(void) { return g_launches.load(); }

sc_status sc_release_stream(sc_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SC_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SC_ERR_CUDA;
    sc_status st = SC_OK;
    HostPipe* hp = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_pipe_mu);
        auto it = g_pipes.find({dev, s});
        if (it != g_pipes.end()) {
            hp = it->second;
            g_pipes.erase(it);
        }
    }
    if (hp) {
        {
            std::lock_guard<std::mutex> lk(hp->mu);  // no sc_scan_host call of this stream still inside
            st = pipe_destroy(*hp, dev);
        }
        delete hp;
    }
    std::lock_guard<std::mutex> lk(g_ws_mu);
    auto it = g_ws.find({dev, s});
    if (it != g_ws.end()) {
        if (it->second.owned && it->second.base && cudaFree(it->second.base) != cudaSuccess) st = SC_ERR_CUDA;
        g_ws.erase(it);
    }
    return st;
}

int sc_debug_last_path(void) { return g_last_path; }

sc_status sc_debug_lookback_stats(sc_stream_t stream, uint64_t* out8) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!out8) return SC_ERR_INVALID;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SC_ERR_CUDA;
    unsigned char* base = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_ws_mu);
        auto it = g_ws.find({dev, s});
        if (it != g_ws.end()) base = it->second.base;
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return SC_ERR_CUDA;
    if (!base) {
        for (int i = 0; i < 8; ++i) out8[i] = 0;
        return SC_OK;
    }
    if (cudaMemcpy(out8, base + kStatsOffset, 64, cudaMemcpyDeviceToHost) != cudaSuccess) return SC_ERR_CUDA;
    if (cudaMemset(base + kStatsOffset, 0, 64) != cudaSuccess) return SC_ERR_CUDA;
    return SC_OK;
}

sc_status sc_set_scan_variant(int variant) {
    if (variant < 0 || variant > max_variant()) return SC_ERR_INVALID;
    g_variant.store(variant);
    return SC_OK;
}

sc_status sc_set_status_stride(int bytes) {
    if (bytes != 0 && bytes != -1 && bytes != 16 && bytes != 32 && bytes != 64 && bytes != 128) return SC_ERR_INVALID;
    g_status_stride.store(bytes);
    return SC_OK;
}

sc_status sc_set_compact_variant(int variant) {
    if (variant < 0 || variant > 7) return SC_ERR_INVALID;
    g_compact_variant.store(variant);
    return SC_OK;
}

sc_status sc_set_radix_variant(int variant) {
    if (variant < 0 || variant >= scg::radix_num_variants()) return SC_ERR_INVALID;
    g_radix_variant.store(variant);
    return SC_OK;
}

sc_status sc_scan_variant_info(int variant, int* threads, int* items, int* loader) {
    if (variant < 0 || variant > max_variant()) return SC_ERR_INVALID;
    const int cfg = tma_cfg_of(variant);
    if (cfg >= 0) {  // persistent TMA kernel: compute threads, 4-byte items per compute thread
        scg::TmaShape sh{0, 0, 0, 0, 1, 2};
        scg::tma_shape(cfg, &sh);
        if (threads) *threads = sh.compute_threads;
        if (items) *items = sh.tile_bytes / 4 / sh.compute_threads;
        if (loader) *loader = 2;
        return SC_OK;
    }
    const scg::ScanShape sh = scg::kShapeSumU32[variant - 1];
    if (threads) *threads = sh.nt;
    if (items) *items = sh.ipt;
    if (loader) *loader = sh.load;
    return SC_OK;
}

sc_status sc_debug_set_lookback(int64_t stall_tile, int64_t delay_tile, uint32_t delay_ns, uint64_t timeout_ns) {
    if (stall_tile < -1 || delay_tile < -1) return SC_ERR_INVALID;
    if (delay_ns > 1000000000u) return SC_ERR_INVALID;
    g_stall_tile.store(stall_tile);
    g_delay_tile.store(delay_tile);
    g_delay_ns.store(delay_ns);
    g_timeout_ns.store(timeout_ns == 0 ? kDefaultTimeoutNs : timeout_ns);
    return SC_OK;
}

}  // extern "C"

// Tile sizes (host side).
namespace scg {
unsigned lookback_stride_words(size_t area, long long units) { return status_stride_words(area, units); }
void lookback_hooks(LookbackCtl* lb) {
    lb->stall_tile = g_stall_tile.load();
    lb->delay_tile = g_delay_tile.load();
    lb->delay_ns = g_delay_ns.load();
    lb->timeout_ns = g_timeout_ns.load();
}

int scan_tile_elems(int op_id, int variant) {
    const ScanShape sh = scan_shape(op_id, variant);
    return sh.nt * sh.ipt;
}
ScanShape scan_shape(int op_id, int variant) {
    switch (op_id) {
    case 0: return (variant >= 0 && variant < kNumSumU32Variants) ? kShapeSumU32[variant] : ScanShape{0, 0, 0};
    case 1: return variant == 0 ? kShapeSumF32 : ScanShape{0, 0, 0};
    case 2: return variant == 0 ? kShapeMaxI32 : ScanShape{0, 0, 0};
    case 3: return variant == 0 ? kShapeAffine : ScanShape{0, 0, 0};
    default:
        if (op_id < kFirstExtraOid || op_id >= OID_COUNT || variant != 0) return ScanShape{0, 0, 0};
        return oid_elem_bytes(op_id) == 8 ? kShapeExtra8 : kShapeExtra4;
    }
}

cudaError_t launch_scan_extra(int oid, const ScanParams& p, bool exclusive, bool segmented, unsigned tma_grid,
                              cudaStream_t s) {
    switch (oid) {
    case OID_PROD_U32: case OID_AND_U32: case OID_OR_U32: case OID_XOR_U32:
        return launch_ops_int32_bits(oid, p, exclusive, segmented, tma_grid, s);
    case OID_MIN_I32: case OID_MAX_U32: case OID_MIN_U32:
        return launch_ops_int32_order(oid, p, exclusive, segmented, tma_grid, s);
    case OID_SUM_U64: case OID_PROD_U64: case OID_AND_U64: case OID_OR_U64: case OID_XOR_U64:
        return launch_ops_int64_bits(oid, p, exclusive, segmented, tma_grid, s);
    case OID_MAX_I64: case OID_MIN_I64: case OID_MAX_U64: case OID_MIN_U64:
        return launch_ops_int64_order(oid, p, exclusive, segmented, tma_grid, s);
    case OID_MAX_F32: case OID_MIN_F32: case OID_SUM_F64:
        return launch_ops_float_a(oid, p, exclusive, segmented, tma_grid, s);
    case OID_MAX_F64: case OID_MIN_F64: case OID_MAXCOUNT_I32:
        return launch_ops_float_b(oid, p, exclusive, segmented, tma_grid, s);
    default: return cudaErrorInvalidValue;
    }
}
}  // namespace scg
