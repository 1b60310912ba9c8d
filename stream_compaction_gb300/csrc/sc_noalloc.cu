// sc_scan_noalloc: the single-pass scan for callers that cannot allocate.
//
// Who needs this: code that runs where device allocation is unavailable or
// forbidden -- for example inside a host callback or a custom allocator's own
// bookkeeping, in a process whose memory pool is owned by another framework
// that does not expose it, or in real-time paths that must not risk the
// device-wide synchronisation a cudaMalloc/cudaFree can cause.  Those callers
// can still provide their input and output buffers, but not the look-back
// workspace that sc_scan_inclusive / sc_scan_exclusive allocate on first use.
//
// Here the workspace is a fixed-size array in the library's own device image
// (`g_noalloc_scratch` below).  Every GPU that loads the library holds one copy
// of it until the process exits.  Nothing in this file calls cudaMalloc,
// cudaFree or any routine that allocates.
#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/sc_scan.h"
#include "sc_launch.h"
#include "sc_shapes.h"

namespace {

// Layout: [0, 8) tile counter, [8, 12) error word, [256, ...) one 16-byte
// look-back status slot per tile (tiles of at least 2048 elements).
constexpr size_t kHeader = 256;
constexpr size_t kSlot = 16;
constexpr long long kMinTile = 2048;
constexpr size_t kScratchBytes = kHeader + kSlot * (SC_NOALLOC_MAX_N / kMinTile);
constexpr unsigned kMaxEpoch = (1u << 30) - 1;
constexpr int kMaxDevices = 64;

// The scratch array.  In host code this name is only a stand-in for the
// device object; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceSlot {
    void* addr = nullptr;     // device address of g_noalloc_scratch on this device (its context at set-up)
    unsigned epoch = 0;       // last epoch used for the status words
    bool ready = false;
};
std::mutex g_mu;
DeviceSlot g_slots[kMaxDevices];

// Once per device, with that device current: look up the device address of
// the scratch array.
sc_status setup(int dev, DeviceSlot** out) {
    if (dev < 0 || dev >= kMaxDevices) return SC_ERR_CUDA;
    DeviceSlot& s = g_slots[dev];
    if (!s.ready) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return SC_ERR_CUDA;
        }
        s.addr = p;
        s.epoch = 0;
        s.ready = true;
    }
    *out = &s;
    return SC_OK;
}

int op_index(sc_dtype d, sc_op o) {
    if (o == SC_SUM && (d == SC_I32 || d == SC_U32)) return 0;
    if (o == SC_SUM && d == SC_F32) return 1;
    if (o == SC_MAX && d == SC_I32) return 2;
    if (o == SC_COMPOSE && d == SC_AFFINE_U32) return 3;
    return -1;
}

}  // namespace

extern "C" sc_status sc_scan_noalloc(sc_dtype dtype, sc_op op, int exclusive, const void* in, void* out, int64_t n,
                                     sc_stream_t stream) {
    if (dtype < SC_I32 || dtype > SC_MAXCOUNT_I32 || op < SC_SUM || op > SC_XOR || n < 0) return SC_ERR_INVALID;
    const int oid = op_index(dtype, op);
    if (oid < 0) return SC_ERR_UNSUPPORTED;
    if (n == 0) return SC_OK;
    if (n > SC_NOALLOC_MAX_N) return SC_ERR_WORKSPACE;  // beyond the fixed scratch
    const size_t eb = dtype == SC_AFFINE_U32 ? 8 : 4;
    const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
    if (!in || !out || a % eb || b % eb) return SC_ERR_INVALID;
    const size_t bytes = (size_t)n * eb;
    if (a != b && a < b + bytes && b < a + bytes) return SC_ERR_INVALID;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;  // the epoch is host state: no capture
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return SC_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return SC_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SC_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceSlot* slot = nullptr;
    sc_status st = setup(dev, &slot);
    if (st != SC_OK) return st;
    unsigned char* base = static_cast<unsigned char*>(slot->addr);

    // The array keeps the previous call's contents.  The tile counter must
    // start at zero; status words of earlier calls carry an older epoch and
    // read as "not yet published", so they need no clearing except when the
    // epoch wraps.  The error word is left alone: it collects every call's
    // failures until sc_scan_noalloc_error reads and clears it.
    // float32 sums carry float-float pairs in one-word statuses with a 7-bit epoch
    const unsigned max_epoch = oid == 1 ? (1u << scg::kFloat2EpochBits) - 1 : kMaxEpoch;
    if (slot->epoch >= max_epoch) {
        if (cudaMemsetAsync(base + kHeader, 0, kScratchBytes - kHeader, s) != cudaSuccess) return SC_ERR_CUDA;
        slot->epoch = 0;
    }
    if (cudaMemsetAsync(base, 0, 8, s) != cudaSuccess) return SC_ERR_CUDA;

    const int tile = scg::scan_tile_elems(oid, 0);
    scg::ScanParams p;
    p.in = in;
    p.out = out;
    p.n = n;
    p.seg_len = 0;
    p.heads = nullptr;
    p.vec_ok = (a % 16 == 0) && (b % 16 == 0);
    p.carry_in = nullptr;
    p.carry_out = nullptr;
    p.lb.status = reinterpret_cast<unsigned long long*>(base + kHeader);
    p.lb.counter = reinterpret_cast<unsigned long long*>(base);
    p.lb.error = reinterpret_cast<unsigned int*>(base + 8);
    p.lb.counter_base = 0;
    p.lb.epoch = ++slot->epoch;
    p.lb.num_tiles = (unsigned)((n + tile - 1) / tile);
    p.lb.static_ids = 0;
    scg::lookback_hooks(&p.lb);  // the time bound, and the test hooks when set
    p.lb.stats = nullptr;
    p.lb.stride_words = scg::lookback_stride_words(kScratchBytes - kHeader, p.lb.num_tiles);
    cudaError_t e;
    switch (oid) {
    case 0: e = scg::launch_scan<scg::OpSumU32>(p, exclusive != 0, false, 0, s); break;
    case 1: e = scg::launch_scan<scg::OpSumF32>(p, exclusive != 0, false, 0, s); break;
    case 2: e = scg::launch_scan<scg::OpMaxI32>(p, exclusive != 0, false, 0, s); break;
    default: e = scg::launch_scan<scg::OpAffineU32>(p, exclusive != 0, false, 0, s); break;
    }
    return e == cudaSuccess ? SC_OK : SC_ERR_CUDA;
}

extern "C" sc_status sc_scan_noalloc_error(sc_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SC_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SC_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (dev < 0 || dev >= kMaxDevices) return SC_ERR_CUDA;
    if (!g_slots[dev].ready) return SC_OK;  // no call on this device yet
    unsigned char* base = static_cast<unsigned char*>(g_slots[dev].addr);
    unsigned int word = 0;
    if (cudaMemcpy(&word, base + 8, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return SC_ERR_CUDA;
    if (word != 0 && cudaMemset(base + 8, 0, sizeof(word)) != cudaSuccess) return SC_ERR_CUDA;
    return (sc_status)word;
}
