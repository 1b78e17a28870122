// decode_noalloc.cu -- split-KV decode for callers that cannot allocate device memory.
//
// attn_decode_splitkv needs a caller-provided workspace.  Some callers have no way to
// provide one: code that runs where cudaMalloc is not allowed or not available to it
// (for example a plugin inside a host framework that owns every device allocation and
// hands out no scratch, or a serving loop that must not allocate after start-up because
// allocation can synchronise the device and stall other streams).  For them this file
// keeps the decode scratch in a fixed array that is part of the library image itself,
// so a call needs nothing beyond its inputs and outputs.
//
// The array is a file-scope __device__ object: every GPU that loads the library reserves
// kNoAllocScratchBytes for it until the process exits.  Host code cannot use the
// array's name as a device address (on the host it names a stand-in), so the device
// address is looked up once per device with cudaGetSymbolAddress while that device is
// current.  That lookup happens inside the first call made on each device; make that
// first call before any stream capture begins.
//
// All calls share the one array and it keeps whatever the previous call left in it.
// The counters that must start at zero are cleared on the stream at the start of every
// call; the partial results need no clearing.  Two calls whose GPU work overlaps (on
// different streams, or on one stream from several host threads without ordering) race
// on the array and produce wrong results: order them on one stream.
#include <cuda_runtime.h>

#include <mutex>

#include "gbattn.h"

namespace {

// Largest scratch a call may need (see attn_decode_workspace_size): 8 MiB covers, for
// example, B = 4 sequences x 64 query heads x 16 splits x d = 128 (about 2.1 MiB).
constexpr size_t kNoAllocScratchBytes = 8u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once per device.
void* scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    static std::mutex mu;
    static void* addr[kMaxDevices] = {nullptr};
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) {
            // the lookup's error is not sticky: clear it so that the caller's next
            // cudaGetLastError() does not report it a second time
            (void)cudaGetLastError();
            return nullptr;
        }
        addr[dev] = ptr;
    }
    return addr[dev];
}

}  // namespace

extern "C" int attn_decode_splitkv_noalloc(const void* q, const void* kcache,
                                           const void* vcache, const int* kv_lens, void* o,
                                           float* lse, int B, int Hq, int Hkv, int Lmax, int d,
                                           float scale, int num_splits, void* stream) {
    // Argument checks first, without touching the device: with no workspace the regular
    // entry point returns GBATTN_ERR_WORKSPACE for valid arguments and launches nothing;
    // any other status names an argument problem.
    const int st = attn_decode_splitkv(q, kcache, vcache, kv_lens, o, lse, B, Hq, Hkv, Lmax, d,
                                       scale, num_splits, nullptr, 0, stream);
    if (st != GBATTN_ERR_WORKSPACE) return st;
    const size_t need = attn_decode_workspace_size(B, Hq, Hkv, Lmax, d, num_splits);
    if (need == 0 || need > kNoAllocScratchBytes) return GBATTN_ERR_WORKSPACE;
    void* scratch = scratch_for_current_device();
    if (scratch == nullptr) return GBATTN_ERR_CUDA;
    return attn_decode_splitkv(q, kcache, vcache, kv_lens, o, lse, B, Hq, Hkv, Lmax, d, scale,
                               num_splits, scratch, kNoAllocScratchBytes, stream);
}
