// decode_noalloc.cu -- split-KV decode for callers that cannot allocate device memory.
//
// blasst_decode needs a caller-provided workspace for the per-split partial
// results whenever it splits the key range.  Some callers have no way to provide
// one: code whose device memory is entirely owned by another allocator (a
// framework's caching pool, a pre-reserved arena) and which may not call
// cudaMalloc itself, or latency-critical serving loops that must not allocate
// between steps.  blasst_decode_noalloc serves them: it passes blasst_decode a
// workspace that lives in this library's own statically sized device array, so
// the call itself allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads this library
// holds it until the process exits.  Its host-side name is only a stand-in, so the
// device address is looked up with cudaGetSymbolAddress, once per device, on the
// first call made with that device current (make that first call before any
// stream capture).  Host threads making their first calls at once each look it up
// and store the same value in an atomic slot.  The cached address does not survive
// cudaDeviceReset.  All calls on a device share the one array: calls whose work
// overlaps on the GPU (different streams, or host threads racing) overwrite each
// other's partial results.  Nothing in it has to start at zero -- each call's split
// pass writes every partial it later merges.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "blasst.h"
#include "kernels.cuh"

namespace {

// 1 Mi floats (4 MiB): room for num_splits * B * Hq * (d + 1) partial values,
// e.g. 2 splits x 64 sequences x 32 heads x (128 + 1) = 528,384.
constexpr size_t kScratchFloats = size_t(1) << 20;
constexpr int kMaxDevices = 64;

}  // namespace

static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

namespace {

void* scratch_address(int* status) {
    static std::atomic<void*> addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = BLASST_ERR_CUDA;
        return nullptr;
    }
    void* cached = addr[dev].load(std::memory_order_acquire);
    if (!cached) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) {
            *status = BLASST_ERR_CUDA;
            return nullptr;
        }
        cached = p;
        addr[dev].store(cached, std::memory_order_release);
    }
    *status = BLASST_OK;
    return cached;
}

}  // namespace

extern "C" size_t blasst_decode_noalloc_scratch_bytes(void) { return kScratchFloats * sizeof(float); }

extern "C" int blasst_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                                     int B, int Hq, int Hkv, int Lkv, int d, float scale, float lambda,
                                     int num_splits, unsigned long long* skipped_tiles_out, unsigned char* skip_map,
                                     float* margins, void* stream) {
    // bad arguments are reported as such before the size check
    const int rc = blasst::decode_args_status(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Lkv, d, scale, lambda,
                                              num_splits, skipped_tiles_out, margins);
    if (rc != BLASST_OK) return rc;
    const size_t need = blasst_decode_workspace_size(B, Hq, Hkv, Lkv, d, num_splits);
    if (need > kScratchFloats * sizeof(float)) return BLASST_ERR_SCRATCH_LIMIT;
    void* ws = nullptr;
    if (need > 0) {
        int st = BLASST_OK;
        ws = scratch_address(&st);
        if (!ws) return st;
    }
    return blasst_decode(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Lkv, d, scale, lambda, num_splits, ws,
                         need > 0 ? kScratchFloats * sizeof(float) : 0, skipped_tiles_out, skip_map, margins,
                         stream);
}
