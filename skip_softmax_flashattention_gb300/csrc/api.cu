// api.cu -- the C ABI declared in include/blasst.h: argument validation, the
// threshold resolution, TMA descriptor encoding and kernel launches.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <initializer_list>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "blasst.h"
#include "kernels.cuh"

// The library's one piece of device state: a sticky status word per device that a
// kernel sets when one of its bounded waits gives up.
__device__ int g_blasst_status = 0;

namespace {

using blasst::kTile;

constexpr unsigned long long kWatchdogNs = 4000000000ull;  // 4 s per wait
constexpr unsigned long long kShortWatchdogNs = 200000ull;  // test flag: 200 us
constexpr int kMaxDevices = 64;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Device address of the status word on the current device, looked up once per device.
// Host threads may make their first calls at the same time: each looks the address up
// and stores the same value, so an atomic slot is all the synchronisation needed.  The
// cached address does not survive cudaDeviceReset (the array moves to a new context).
int* status_word() {
    static std::atomic<int*> ptrs[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int* cached = ptrs[dev].load(std::memory_order_acquire);
    if (!cached) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_blasst_status) != cudaSuccess || !p) return nullptr;
        cached = static_cast<int*>(p);
        ptrs[dev].store(cached, std::memory_order_release);
    }
    return cached;
}

// True iff every pointer is device memory of the current device.  The cluster
// kernels (MLA decode above 64 heads, GQA decode with 128 heads per KV head) multicast
// their TMA key loads to the CTAs of a cluster; those loads must read this GPU's own
// memory, so memory of another GPU (peer-mapped or imported), managed memory and host
// memory are refused.  A failed query counts as a refusal.
bool local_device_memory(std::initializer_list<const void*> ptrs) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    for (const void* p : ptrs) {
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
            (void)cudaGetLastError();
            return false;
        }
        if (a.type != cudaMemoryTypeDevice || a.device != dev) return false;
    }
    return true;
}

// [Z][L][d] bf16 viewed as a 3-D tensor (d fastest); boxes of 64 columns x 128 rows,
// 128-byte swizzle, zero fill outside [0, L).
bool encode_3d(CUtensorMap* map, const void* base, int d, int L, long long Z) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)L, (cuuint64_t)Z};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)L * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// [Z][L][d] bf16 as a 3-D tensor with boxes of 64 columns x `rows` rows (the latent
// page pool of MLA decode: Z = 1, L = num_pages * page_size rows of d values).
bool encode_rows(CUtensorMap* map, const void* base, int d, long long L, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)L, 1};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)L * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 4-D map over a page pool of bf16 K or V, box = 64 columns x `rows` keys of one
// head of one page.  Dimensions are ordered by stride:
//   key-major pool [page][key][head][d]: (d, head, key, page)
//   head-major pool [page][head][key][d]: (d, key, head, page)
bool encode_pages(CUtensorMap* map, const void* base, int d, int page_size, int Hkv, long long num_pages,
                  int token_major, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t e = 2;
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4];
    if (token_major) {
        dims[0] = d; dims[1] = Hkv; dims[2] = page_size; dims[3] = num_pages;
        strides[0] = d * e; strides[1] = (cuuint64_t)Hkv * d * e; strides[2] = (cuuint64_t)page_size * Hkv * d * e;
        box[0] = 64; box[1] = 1; box[2] = rows; box[3] = 1;
    } else {
        dims[0] = d; dims[1] = page_size; dims[2] = Hkv; dims[3] = num_pages;
        strides[0] = d * e; strides[1] = (cuuint64_t)page_size * d * e; strides[2] = (cuuint64_t)Hkv * page_size * d * e;
        box[0] = 64; box[1] = rows; box[2] = 1; box[3] = 1;
    }
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Queries [B][H][d] bf16 as a 3-D tensor, boxes of 64 columns x `rows` heads of one
// sequence; heads past H and columns past d read as zeros.
bool encode_heads(CUtensorMap* map, const void* base, int d, int H, int B, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool lambda_ok(float lambda) { return std::isfinite(lambda) && lambda >= 0.f && lambda <= 1.f; }

bool scale_ok(float scale) { return std::isfinite(scale) && scale > 0.f; }

struct Thresholds {
    float c_log2, thr_raw, lazy_raw;
};

// Convert (scale, lambda) into the kernels' raw-score units: a score s = scale*x,
// the test m~ - m < ln(lambda) becomes x~ - x_m < ln(lambda)/scale.
Thresholds thresholds(float scale, float lambda) {
    const double log2e = 1.4426950408889634;
    Thresholds t;
    t.c_log2 = (float)((double)scale * log2e);
    t.thr_raw = lambda > 0.f ? (float)(std::log((double)lambda) / (double)scale) : -INFINITY;
    t.lazy_raw = (float)(8.0 / ((double)scale * log2e));
    return t;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? BLASST_OK : BLASST_ERR_CUDA; }

// One decode CTA fits per SM.  Take the fewest splits whose `units` x splits CTAs
// fill the last wave to at least 90%; more splits restart the running max more often.
int plan_splits(long long units, int nT, int* out) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return BLASST_ERR_CUDA;
    int best = 1;
    double best_eff = 0.0;
    for (int S = 1; S <= nT && S <= 64; ++S) {
        const double waves = (double)(units * S) / sms;
        const double eff = waves / std::ceil(waves);
        if (eff >= 0.9) {
            best = S;
            best_eff = eff;
            break;
        }
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = S;
        }
    }
    *out = best;
    return BLASST_OK;
}

bool page_size_ok(int page_size) {
    // a 128-key tile is whole pages or lies inside one page
    return page_size == 8 || page_size == 16 || page_size == 32 || page_size == 64 ||
           (page_size > 0 && page_size % kTile == 0);
}

}  // namespace

namespace blasst {

int decode_args_status(const void* q, const void* k_cache, const void* v_cache, const void* o, const float* lse,
                       int B, int Hq, int Hkv, int Lkv, int d, float scale, float lambda, int num_splits,
                       const unsigned long long* skipped_tiles_out, const float* margins) {
    if (!q || !k_cache || !v_cache || !o) return BLASST_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || Lkv < 1 || Hq % Hkv != 0) return BLASST_ERR_INVALID_ARG;
    if (!scale_ok(scale) || !lambda_ok(lambda)) return BLASST_ERR_INVALID_ARG;
    const int nT = (Lkv + kTile - 1) / kTile;
    if (num_splits < 1 || num_splits > nT) return BLASST_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if (d != 64 && d != 128) return BLASST_ERR_UNSUPPORTED;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16 && G != 32 && G != 64 && G != 128)
        return BLASST_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o)) return BLASST_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(margins) & 3u) ||
        (reinterpret_cast<uintptr_t>(skipped_tiles_out) & 7u))
        return BLASST_ERR_UNSUPPORTED;
    if (Hkv > 65535 || B > 65535) return BLASST_ERR_UNSUPPORTED;
    return BLASST_OK;
}

}  // namespace blasst

extern "C" {

int blasst_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                   int Lq, int Lkv, int d, int causal, float scale, float lambda,
                   unsigned long long* skipped_tiles_out, void* stream) {
    return blasst_prefill_ex(q, k, v, o, lse, B, Hq, Hkv, Lq, Lkv, d, causal, scale, lambda, skipped_tiles_out,
                             nullptr, nullptr, 0u, stream);
}

static int prefill_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Lq, int Lkv, int d, int causal, int window, float scale, float lambda,
                        unsigned long long* skipped_tiles_out, unsigned char* skip_map, float* margins,
                        unsigned flags, void* stream);

int blasst_prefill_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                      int Hkv, int Lq, int Lkv, int d, int causal, float scale, float lambda,
                      unsigned long long* skipped_tiles_out, unsigned char* skip_map, float* margins,
                      unsigned flags, void* stream) {
    return prefill_impl(q, k, v, o, lse, B, Hq, Hkv, Lq, Lkv, d, causal, 0, scale, lambda, skipped_tiles_out,
                        skip_map, margins, flags, stream);
}

int blasst_prefill_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                          int Hkv, int Lq, int Lkv, int d, int window, float scale, float lambda,
                          unsigned long long* skipped_tiles_out, unsigned char* skip_map, float* margins,
                          unsigned flags, void* stream) {
    if (window < 1) return BLASST_ERR_INVALID_ARG;
    if (flags & (BLASST_PREFILL_P_VIA_SMEM | BLASST_PREFILL_ONE_QTILE | BLASST_PREFILL_WIDE))
        return BLASST_ERR_UNSUPPORTED;  // the window is built into the default kernel only
    return prefill_impl(q, k, v, o, lse, B, Hq, Hkv, Lq, Lkv, d, 1, window, scale, lambda, skipped_tiles_out,
                        skip_map, margins, flags, stream);
}

static int prefill_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Lq, int Lkv, int d, int causal, int window, float scale, float lambda,
                        unsigned long long* skipped_tiles_out, unsigned char* skip_map, float* margins,
                        unsigned flags, void* stream) {
    if (!q || !k || !v || !o) return BLASST_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lkv < 1 || Hq % Hkv != 0) return BLASST_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return BLASST_ERR_INVALID_ARG;
    if (!scale_ok(scale) || !lambda_ok(lambda)) return BLASST_ERR_INVALID_ARG;
    const unsigned known = BLASST_PREFILL_ELIDE_V | BLASST_PREFILL_P_VIA_SMEM | BLASST_PREFILL_ONE_QTILE |
                           BLASST_PREFILL_WIDE | BLASST_FLAG_TEST_SHORT_WATCHDOG;
    if (flags & ~known) return BLASST_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return BLASST_ERR_UNSUPPORTED;
    if ((flags & BLASST_PREFILL_ELIDE_V) &&
        (flags & (BLASST_PREFILL_P_VIA_SMEM | BLASST_PREFILL_ONE_QTILE | BLASST_PREFILL_WIDE)))
        return BLASST_ERR_UNSUPPORTED;  // V elision is built into the default kernel only
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return BLASST_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(margins) & 3u) ||
        (reinterpret_cast<uintptr_t>(skipped_tiles_out) & 7u))
        return BLASST_ERR_UNSUPPORTED;
    if (Hq > 65535 || B > 65535) return BLASST_ERR_UNSUPPORTED;
    const long long nQ = (Lq + kTile - 1) / kTile, nK = (Lkv + kTile - 1) / kTile;
    if (nQ * B * Hq > 0x7fffffffLL) return BLASST_ERR_UNSUPPORTED;  // one-dimensional grid

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int* status = status_word();
    if (!status) return BLASST_ERR_CUDA;
    CUtensorMap tq, tk, tv;
    if (!encode_3d(&tq, q, d, Lq, (long long)B * Hq) || !encode_3d(&tk, k, d, Lkv, (long long)B * Hkv) ||
        !encode_3d(&tv, v, d, Lkv, (long long)B * Hkv))
        return BLASST_ERR_CUDA;

    const long long map_n = (long long)B * Hq * nQ * nK;
    if (skipped_tiles_out && cudaMemsetAsync(skipped_tiles_out, 0, sizeof(unsigned long long), st) != cudaSuccess)
        return BLASST_ERR_CUDA;
    if (skip_map && cudaMemsetAsync(skip_map, 2, (size_t)map_n, st) != cudaSuccess) return BLASST_ERR_CUDA;
    if (margins && cudaMemsetAsync(margins, 0xFF, (size_t)map_n * sizeof(float), st) != cudaSuccess)
        return BLASST_ERR_CUDA;

    const Thresholds t = thresholds(scale, lambda);
    blasst::PrefillParams p{};
    p.o = o;
    p.lse = lse;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Lq = Lq; p.Lkv = Lkv; p.causal = causal;
    p.nQ = (int)nQ; p.nK = (int)nK;
    p.c_log2 = t.c_log2;
    p.scale = scale;
    p.thr_raw = t.thr_raw;
    p.lazy_raw = t.lazy_raw;
    p.skipped = skipped_tiles_out;
    p.skip_map = skip_map;
    p.margins = margins;
    p.status = status;
    p.watchdog_ns = (flags & BLASST_FLAG_TEST_SHORT_WATCHDOG) ? kShortWatchdogNs : kWatchdogNs;
    p.elide_v = (flags & BLASST_PREFILL_ELIDE_V) ? 1 : 0;
    p.window = window;
    p.test_stall = (flags & BLASST_FLAG_TEST_SHORT_WATCHDOG) ? 1 : 0;
    // CTA order: under a causal mask the query tiles differ in work, so hand them out
    // longest-first within bands of whole K/V-head groups whose K and V take at most an
    // eighth of L2, so that the streaming Q and O do not evict them (measured on the
    // causal 16k GQA prefill: 201 MB of DRAM reads, the algorithmic Q + K + V, against
    // 280 MB with bands of seven groups); without a mask every tile costs the same and
    // head-major order is kept.
    p.band = 1;
    if (causal) {
        int dev = 0, l2 = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
            return BLASST_ERR_CUDA;
        const long long kv_head_bytes = 2LL * Lkv * d * 2;
        const long long groups = std::max(1LL, (long long)(l2 / 8) / kv_head_bytes);
        p.band = (int)std::min<long long>((long long)B * Hq, groups * (Hq / Hkv));
    }
    const blasst::PrefillVariant var = (flags & BLASST_PREFILL_P_VIA_SMEM) ? blasst::PrefillVariant::kOneTilePSmem
                                       : (flags & BLASST_PREFILL_ONE_QTILE) ? blasst::PrefillVariant::kOneTilePTmem
                                       : (flags & BLASST_PREFILL_WIDE)      ? blasst::PrefillVariant::kWide
                                                                            : blasst::PrefillVariant::kTwoTiles;
    return cuda_status(blasst::launch_prefill(tq, tk, tv, p, d, var, st));
}

int blasst_decode_num_splits(int B, int Hq, int Hkv, int Lkv, int d, int requested, int* out) {
    if (!out || B < 1 || Hq < 1 || Hkv < 1 || Lkv < 1 || d < 1 || Hq % Hkv != 0 || requested < 0)
        return BLASST_ERR_INVALID_ARG;
    const int nT = (Lkv + kTile - 1) / kTile;
    if (requested > 0) {
        if (requested > nT) return BLASST_ERR_INVALID_ARG;
        *out = requested;
        return BLASST_OK;
    }
    // G > 64: a cluster of G / 64 CTAs per (sequence, KV head, split)
    const int G = Hq / Hkv;
    return plan_splits((long long)B * Hkv * (G > 64 ? G / 64 : 1), nT, out);
}

size_t blasst_decode_workspace_size(int B, int Hq, int Hkv, int Lkv, int d, int num_splits) {
    (void)Hkv;
    (void)Lkv;
    if (B < 1 || Hq < 1 || d < 1 || num_splits <= 1) return 0;
    const size_t o_bytes = (size_t)num_splits * B * Hq * d * sizeof(float);
    const size_t l_bytes = (size_t)num_splits * B * Hq * sizeof(float);
    return ((o_bytes + 255) & ~size_t(255)) + l_bytes;
}

static int run_decode(const CUtensorMap& tk, const CUtensorMap& tv, blasst::DecodeParams& p, const void* q, void* o,
               float* lse, int B, int Hq, int Hkv, int Lkv, int d, float scale, float lambda, int num_splits,
               void* workspace, unsigned long long* skipped_tiles_out, unsigned char* skip_map, float* margins,
               void* stream);

int blasst_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B, int Hq,
                  int Hkv, int Lkv, int d, float scale, float lambda, int num_splits, void* workspace,
                  size_t workspace_bytes, unsigned long long* skipped_tiles_out, unsigned char* skip_map,
                  float* margins, void* stream) {
    const int rc = blasst::decode_args_status(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Lkv, d, scale, lambda,
                                              num_splits, skipped_tiles_out, margins);
    if (rc != BLASST_OK) return rc;
    const size_t need = blasst_decode_workspace_size(B, Hq, Hkv, Lkv, d, num_splits);
    if (num_splits > 1) {
        if (!workspace) return BLASST_ERR_INVALID_ARG;
        if (workspace_bytes < need) return BLASST_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned16(workspace)) return BLASST_ERR_UNSUPPORTED;
    }
    // 128 heads per KV head run as clusters whose key loads are multicast
    if (Hq / Hkv > 64 && !local_device_memory({q, k_cache, v_cache})) return BLASST_ERR_UNSUPPORTED;

    CUtensorMap tk, tv;
    if (!encode_3d(&tk, k_cache, d, Lkv, (long long)B * Hkv) || !encode_3d(&tv, v_cache, d, Lkv, (long long)B * Hkv))
        return BLASST_ERR_CUDA;
    blasst::DecodeParams p{};
    return run_decode(tk, tv, p, q, o, lse, B, Hq, Hkv, Lkv, d, scale, lambda, num_splits, workspace,
                      skipped_tiles_out, skip_map, margins, stream);
}

// The part of blasst_decode and blasst_decode_paged after validation: output
// initialisation, parameters, the split pass and the merge.  `p` carries the
// form-specific fields (page table, lengths) on entry.
static int run_decode(const CUtensorMap& tk, const CUtensorMap& tv, blasst::DecodeParams& p, const void* q, void* o,
               float* lse, int B, int Hq, int Hkv, int Lkv, int d, float scale, float lambda, int num_splits,
               void* workspace, unsigned long long* skipped_tiles_out, unsigned char* skip_map, float* margins,
               void* stream) {
    const int nT = (Lkv + kTile - 1) / kTile;
    const int G = Hq / Hkv;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int* status = status_word();
    if (!status) return BLASST_ERR_CUDA;
    const long long map_n = (long long)B * Hkv * nT;
    if (skipped_tiles_out && cudaMemsetAsync(skipped_tiles_out, 0, sizeof(unsigned long long), st) != cudaSuccess)
        return BLASST_ERR_CUDA;
    if (skip_map && cudaMemsetAsync(skip_map, 2, (size_t)map_n, st) != cudaSuccess) return BLASST_ERR_CUDA;
    if (margins && cudaMemsetAsync(margins, 0xFF, (size_t)map_n * sizeof(float), st) != cudaSuccess)
        return BLASST_ERR_CUDA;

    const Thresholds t = thresholds(scale, lambda);
    p.q = static_cast<const uint16_t*>(q);
    p.o = o;
    p.lse = lse;
    const size_t o_bytes = (size_t)num_splits * B * Hq * d * sizeof(float);
    p.o_part = num_splits > 1 ? static_cast<float*>(workspace) : nullptr;
    p.lse_part = num_splits > 1
                     ? reinterpret_cast<float*>(static_cast<char*>(workspace) + ((o_bytes + 255) & ~size_t(255)))
                     : nullptr;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Lkv = Lkv; p.G = G; p.nK = nT; p.S = num_splits; p.d = d;
    p.c_log2 = t.c_log2;
    p.scale = scale;
    p.thr_raw = t.thr_raw;
    p.lazy_raw = t.lazy_raw;
    p.skipped = skipped_tiles_out;
    p.skip_map = skip_map;
    p.margins = margins;
    p.status = status;
    p.watchdog_ns = kWatchdogNs;
    // more than 16 query heads per KV head: the wide-group kernel (contiguous cache)
    cudaError_t e;
    if (G > 16 && !p.page_table) {
        CUtensorMap tq;
        if (!encode_heads(&tq, q, d, Hq, B, blasst::mla_heads_per_cta(G))) return BLASST_ERR_CUDA;
        e = blasst::launch_wide_decode(tk, tv, tq, p, st);
    } else {
        e = blasst::launch_decode(tk, tv, p, d, st);
    }
    if (e != cudaSuccess) return BLASST_ERR_CUDA;
    if (num_splits > 1) {
        blasst::CombineParams c{};
        c.o_part = p.o_part;
        c.lse_part = p.lse_part;
        c.o = o;
        c.lse = lse;
        c.B = B; c.Hq = Hq; c.S = num_splits; c.d = d;
        e = blasst::launch_combine(c, st);
    }
    return cuda_status(e);
}

int blasst_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* page_table,
                        const int* seq_lens, void* o, float* lse, int B, int Hq, int Hkv, int max_kv_len,
                        int window, int d, int num_pages, int page_size, int max_pages_per_seq, int token_major,
                        float scale, float lambda, int num_splits, void* workspace, size_t workspace_bytes,
                        unsigned long long* skipped_tiles_out, unsigned char* skip_map, float* margins,
                        void* stream) {
    if (!q || !k_pages || !v_pages || !page_table || !o) return BLASST_ERR_INVALID_ARG;
    if (window < 0) return BLASST_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || max_kv_len < 1 || Hq % Hkv != 0) return BLASST_ERR_INVALID_ARG;
    if (num_pages < 1 || page_size < 1 || (token_major != 0 && token_major != 1)) return BLASST_ERR_INVALID_ARG;
    if ((long long)max_pages_per_seq * page_size < max_kv_len) return BLASST_ERR_INVALID_ARG;
    if (!scale_ok(scale) || !lambda_ok(lambda)) return BLASST_ERR_INVALID_ARG;
    const int nT = (max_kv_len + kTile - 1) / kTile;
    if (num_splits < 1 || num_splits > nT) return BLASST_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if (d != 64 && d != 128) return BLASST_ERR_UNSUPPORTED;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return BLASST_ERR_UNSUPPORTED;
    if (!page_size_ok(page_size)) return BLASST_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o)) return BLASST_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(margins) & 3u) ||
        (reinterpret_cast<uintptr_t>(page_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(skipped_tiles_out) & 7u))
        return BLASST_ERR_UNSUPPORTED;
    if (Hkv > 65535 || B > 65535) return BLASST_ERR_UNSUPPORTED;
    const size_t need = blasst_decode_workspace_size(B, Hq, Hkv, max_kv_len, d, num_splits);
    if (num_splits > 1) {
        if (!workspace) return BLASST_ERR_INVALID_ARG;
        if (workspace_bytes < need) return BLASST_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned16(workspace)) return BLASST_ERR_UNSUPPORTED;
    }
    const int rows = page_size < kTile ? page_size : kTile;
    CUtensorMap tk, tv;
    if (!encode_pages(&tk, k_pages, d, page_size, Hkv, num_pages, token_major, rows) ||
        !encode_pages(&tv, v_pages, d, page_size, Hkv, num_pages, token_major, rows))
        return BLASST_ERR_CUDA;
    blasst::DecodeParams p{};
    p.seq_lens = seq_lens;
    p.page_table = page_table;
    p.max_pages = max_pages_per_seq;
    p.num_pages = num_pages;
    p.page_size = page_size;
    p.rows_per_box = rows;
    p.token_major = token_major;
    p.window = window;
    return run_decode(tk, tv, p, q, o, lse, B, Hq, Hkv, max_kv_len, d, scale, lambda, num_splits, workspace,
                      skipped_tiles_out, skip_map, margins, stream);
}

int blasst_mla_decode_num_splits(int B, int Hq, int max_kv_len, int requested, int* out) {
    if (!out || B < 1 || Hq < 1 || max_kv_len < 1 || requested < 0) return BLASST_ERR_INVALID_ARG;
    const int nT = (max_kv_len + kTile - 1) / kTile;
    if (requested > 0) {
        if (requested > nT) return BLASST_ERR_INVALID_ARG;
        *out = requested;
        return BLASST_OK;
    }
    // one CTA per (sequence, split), a cluster of Hq / 64 of them above 64 heads
    return plan_splits((long long)B * (Hq > 64 ? Hq / 64 : 1), nT, out);
}

size_t blasst_mla_decode_workspace_size(int B, int Hq, int max_kv_len, int num_splits) {
    return blasst_decode_workspace_size(B, Hq, 1, max_kv_len, blasst::kMlaDv, num_splits);
}

int blasst_mla_decode(const void* q, const void* kv, const int* page_table, const int* seq_lens, void* o,
                      float* lse, int B, int Hq, int max_kv_len, int dk, int dv, int num_pages, int page_size,
                      int max_pages_per_seq, float scale, float lambda, int num_splits, void* workspace,
                      size_t workspace_bytes, unsigned long long* skipped_tiles_out, unsigned char* skip_map,
                      float* margins, void* stream) {
    if (!q || !kv || !o) return BLASST_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || max_kv_len < 1 || dk < 1 || dv < 1) return BLASST_ERR_INVALID_ARG;
    if (!scale_ok(scale) || !lambda_ok(lambda)) return BLASST_ERR_INVALID_ARG;
    if (page_table) {
        if (num_pages < 1 || page_size < 1 || max_pages_per_seq < 1) return BLASST_ERR_INVALID_ARG;
        if ((long long)max_pages_per_seq * page_size < max_kv_len) return BLASST_ERR_INVALID_ARG;
    }
    const int nT = (max_kv_len + kTile - 1) / kTile;
    if (num_splits < 1 || num_splits > nT) return BLASST_ERR_INVALID_ARG;
    if (dk != blasst::kMlaDk || dv != blasst::kMlaDv) return BLASST_ERR_UNSUPPORTED;
    if (Hq != 1 && Hq != 2 && Hq != 4 && Hq != 8 && Hq != 16 && Hq != 32 && Hq != 64 && Hq != 128)
        return BLASST_ERR_UNSUPPORTED;
    if (page_table && !page_size_ok(page_size)) return BLASST_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(o)) return BLASST_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(margins) & 3u) ||
        (reinterpret_cast<uintptr_t>(page_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(skipped_tiles_out) & 7u))
        return BLASST_ERR_UNSUPPORTED;
    if (B > 65535) return BLASST_ERR_UNSUPPORTED;
    const size_t need = blasst_mla_decode_workspace_size(B, Hq, max_kv_len, num_splits);
    if (num_splits > 1) {
        if (!workspace) return BLASST_ERR_INVALID_ARG;
        if (workspace_bytes < need) return BLASST_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned16(workspace)) return BLASST_ERR_UNSUPPORTED;
    }
    // above 64 heads the CTAs of a cluster share key loads by multicast
    if (Hq > 64 && !local_device_memory({q, kv})) return BLASST_ERR_UNSUPPORTED;
    CUtensorMap tkv, tq;
    const int rows = page_size < kTile ? page_size : kTile;
    // pool rows, and the row past the last page that an out-of-range index reads, fit an int
    if (page_table && ((long long)num_pages + 1) * page_size > 0x7fffffffLL - kTile) return BLASST_ERR_UNSUPPORTED;
    if (page_table ? !encode_rows(&tkv, kv, dk, (long long)num_pages * page_size, rows)
                   : !encode_3d(&tkv, kv, dk, max_kv_len, B))
        return BLASST_ERR_CUDA;
    if (!encode_heads(&tq, q, dk, Hq, B, blasst::mla_heads_per_cta(Hq > 64 ? 64 : Hq))) return BLASST_ERR_CUDA;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int* status = status_word();
    if (!status) return BLASST_ERR_CUDA;
    const long long map_n = (long long)B * nT;
    if (skipped_tiles_out && cudaMemsetAsync(skipped_tiles_out, 0, sizeof(unsigned long long), st) != cudaSuccess)
        return BLASST_ERR_CUDA;
    if (skip_map && cudaMemsetAsync(skip_map, 2, (size_t)map_n, st) != cudaSuccess) return BLASST_ERR_CUDA;
    if (margins && cudaMemsetAsync(margins, 0xFF, (size_t)map_n * sizeof(float), st) != cudaSuccess)
        return BLASST_ERR_CUDA;

    const Thresholds t = thresholds(scale, lambda);
    blasst::DecodeParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.o = o;
    p.lse = lse;
    const size_t o_bytes = (size_t)num_splits * B * Hq * dv * sizeof(float);
    p.o_part = num_splits > 1 ? static_cast<float*>(workspace) : nullptr;
    p.lse_part = num_splits > 1
                     ? reinterpret_cast<float*>(static_cast<char*>(workspace) + ((o_bytes + 255) & ~size_t(255)))
                     : nullptr;
    p.B = B; p.Hq = Hq; p.Hkv = 1; p.Lkv = max_kv_len; p.G = Hq; p.nK = nT; p.S = num_splits;
    p.c_log2 = t.c_log2;
    p.scale = scale;
    p.thr_raw = t.thr_raw;
    p.lazy_raw = t.lazy_raw;
    p.skipped = skipped_tiles_out;
    p.skip_map = skip_map;
    p.margins = margins;
    p.status = status;
    p.watchdog_ns = kWatchdogNs;
    p.seq_lens = seq_lens;
    p.page_table = page_table;
    p.max_pages = max_pages_per_seq;
    p.num_pages = num_pages;
    p.page_size = page_size;
    p.rows_per_box = rows;
    p.token_major = 1;
    cudaError_t e = blasst::launch_mla_decode(tkv, tq, p, st);
    if (e != cudaSuccess) return BLASST_ERR_CUDA;
    if (num_splits > 1) {
        blasst::CombineParams c{};
        c.o_part = p.o_part;
        c.lse_part = p.lse_part;
        c.o = o;
        c.lse = lse;
        c.B = B; c.Hq = Hq; c.S = num_splits; c.d = dv;
        e = blasst::launch_combine(c, st);
    }
    return cuda_status(e);
}

int blasst_lambda(int mode, double threshold, double a, double b, double target_sparsity, long long Lkv,
                  double* lambda_out) {
    if (!lambda_out || Lkv < 1) return BLASST_ERR_INVALID_ARG;
    double factor;
    if (mode == 0) {
        if (!std::isfinite(threshold) || threshold < 0.0) return BLASST_ERR_INVALID_ARG;
        factor = threshold * (double)Lkv;  // threshold_scale_factor = threshold * max_kv_len
    } else if (mode == 1) {
        if (!std::isfinite(a) || !std::isfinite(b)) return BLASST_ERR_NO_CALIBRATION;
        if (!std::isfinite(target_sparsity) || target_sparsity < 0.0 || target_sparsity > 1.0 || a < 0.0)
            return BLASST_ERR_INVALID_ARG;
        factor = a * std::exp(b * target_sparsity);  // threshold_scale_factor = a * exp(b * s)
    } else {
        return BLASST_ERR_INVALID_ARG;
    }
    const double lam = mode == 0 ? threshold : factor / (double)Lkv;  // lambda = factor / max_kv_len
    if (!std::isfinite(lam)) return BLASST_ERR_INVALID_ARG;
    *lambda_out = lam;
    return lam > 1.0 ? BLASST_WARN_LAMBDA_GE_1 : BLASST_OK;
}

int blasst_device_status(int clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return BLASST_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_blasst_status, sizeof(int)) != cudaSuccess) return BLASST_ERR_CUDA;
    if (clear && v) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_blasst_status, &zero, sizeof(int)) != cudaSuccess) return BLASST_ERR_CUDA;
    }
    if (v & 2) return BLASST_ERR_CUDA;  // a kernel found its shared memory misaligned
    if (v & 1) return BLASST_ERR_TIMEOUT;
    return v ? BLASST_ERR_PAGE_TABLE : BLASST_OK;
}

const char* blasst_status_string(int status) {
    switch (status) {
        case BLASST_OK: return "ok";
        case BLASST_WARN_LAMBDA_GE_1: return "lambda from the calibration curve exceeds 1";
        case BLASST_ERR_INVALID_ARG: return "invalid argument";
        case BLASST_ERR_UNSUPPORTED: return "unsupported configuration";
        case BLASST_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case BLASST_ERR_CUDA: return "CUDA error";
        case BLASST_ERR_TIMEOUT: return "device wait timed out";
        case BLASST_ERR_PAGE_TABLE: return "page table entry or sequence length out of range (read as zeros / clamped)";
        case BLASST_ERR_NO_CALIBRATION: return "target sparsity requested without calibration coefficients; use a threshold";
        case BLASST_ERR_SCRATCH_LIMIT: return "decode partials exceed the library's static scratch (use blasst_decode with a workspace)";
        default: return "unknown status";
    }
}

}  // extern "C"
