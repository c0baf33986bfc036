// kernels.cuh -- launch-side view of the prefill, decode and combine kernels:
// parameter blocks and launcher declarations shared by the C ABI (api.cu) and
// the kernel translation units.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace blasst {

constexpr int kTile = 128;  // B_r = B_c = 128

struct PrefillParams {
    void* o;                  // bf16 [B,Hq,Lq,d]
    float* lse;               // [B,Hq,Lq] or null
    int B, Hq, Hkv, Lq, Lkv, causal;
    int nQ, nK;
    float c_log2;             // scale * log2(e): raw score -> log2 units
    float scale;              // raw score -> natural-log units
    float thr_raw;            // ln(lambda) / scale (-inf when lambda == 0)
    float lazy_raw;           // reference max is moved only when the max grows by more than this
    unsigned long long* skipped;
    unsigned char* skip_map;  // [B,Hq,nQ,nK] or null
    float* margins;           // [B,Hq,nQ,nK] or null
    int* status;              // device status word
    unsigned long long watchdog_ns;
    int elide_v;
    int test_stall;           // test only: the MMA issuer first waits on a barrier nothing arrives on
    int band;                 // (b, h) pairs per scheduling band, see prefill_cta_coords
    int window;               // > 0 (causal only): row r sees keys r' - window < c <= r', r' = r + Lkv - Lq
};

// Position of this CTA in a one-dimensional prefill grid of nunits * B * Hq CTAs.
// The (b, h) pairs are cut into bands of p.band consecutive pairs (b * Hq + h order,
// so the query heads that share a K/V head sit together); a band's CTAs are handed
// out unit-major -- unit 0 of every pair in the band, then unit 1, ... -- and bands
// follow one another.  With units numbered heaviest first (causal mask), a band
// then runs longest-first, which evens out the finish times of the SMs, while the
// K/V the band reads at once stays small enough for L2.  band == 1 is head-major.
__device__ __forceinline__ void prefill_cta_coords(const PrefillParams& p, int nunits, int& unit, int& b, int& h) {
    const int nbh = p.B * p.Hq;
    const int lin = (int)blockIdx.x;
    const int per_band = p.band * nunits;
    const int bi = lin / per_band;
    const int r = lin - bi * per_band;
    const int bh0 = bi * p.band;
    const int nb = min(p.band, nbh - bh0);
    unit = r / nb;
    const int bh = bh0 + (r - unit * nb);
    b = bh / p.Hq;
    h = bh - b * p.Hq;
}

struct DecodeParams {
    const uint16_t* q;        // bf16 [B,Hq,d]
    void* o;                  // bf16 [B,Hq,d]
    float* lse;               // [B,Hq] or null
    float* o_part;            // [S,B,Hq,d] (S > 1)
    float* lse_part;          // [S,B,Hq]   (S > 1)
    int B, Hq, Hkv, Lkv, G, nK, S;
    int d;                    // head dim of q, k, v, o (GQA decode: 64 or 128; the kernel pads to 128)
    float c_log2, scale, thr_raw, lazy_raw;
    unsigned long long* skipped;
    unsigned char* skip_map;  // [B,Hkv,nK] or null
    float* margins;           // [B,Hkv,nK] or null
    int* status;
    unsigned long long watchdog_ns;
    // Per-sequence key counts and paged K/V (blasst_decode_paged); null / 0 otherwise.
    const int* seq_lens;      // [B]: keys of sequence b (clamped to [0, Lkv]); null: every sequence has Lkv
    const int* page_table;    // [B, max_pages]: physical page of each page_size-key page of sequence b
    int max_pages, num_pages, page_size;
    int rows_per_box;         // keys per TMA box: min(page_size, 128)
    int token_major;          // 1: pool [page][key][head][d]; 0: pool [page][head][key][d]
    int window;               // > 0: only the last `window` keys of each sequence
};

struct CombineParams {
    const float* o_part;
    const float* lse_part;
    void* o;
    float* lse;
    int B, Hq, S, d;
};

// Prefill kernel variants (identical results):
//   kTwoTiles       two 128-row query tiles per CTA, one softmax thread per row (default)
//   kWide           two 128-row query tiles per CTA, two softmax threads per row
//   kOneTilePTmem   one query tile per CTA, S double-buffered, P in TMEM
//   kOneTilePSmem   one query tile per CTA, S double-buffered, P staged in shared memory
enum class PrefillVariant { kWide, kTwoTiles, kOneTilePTmem, kOneTilePSmem };

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int d, PrefillVariant v, cudaStream_t stream);
cudaError_t launch_prefill_wide(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const PrefillParams& p, int d, cudaStream_t stream);
cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, int d,
                          cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);
// MLA decode (absorbed form): rows of kMlaDk values, values = their first kMlaDv.
// DecodeParams carries Hq = G = the query heads (1-128), Hkv = 1, d = kMlaDk.
constexpr int kMlaDk = 576, kMlaDv = 512;
// Query heads one CTA of the MLA / wide-group kernel holds (the MMA N) for G heads per
// KV head; the query tensor map's boxes are this many rows high.
__host__ __device__ constexpr int mla_heads_per_cta(int G) { return G <= 16 ? 16 : G <= 32 ? 32 : 64; }
// tq: the queries [B][Hq][d] as a 3-D map, boxes of 64 columns x mla_heads_per_cta(G) heads.
cudaError_t launch_mla_decode(const CUtensorMap& tkv, const CUtensorMap& tq, const DecodeParams& p,
                              cudaStream_t stream);
// GQA/MQA decode with G = 32, 64 or 128 query heads per KV head (contiguous cache, d 64 or
// 128), on the MLA kernel's wide-group machinery with separate K and V tensors.
cudaError_t launch_wide_decode(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                               const DecodeParams& p, cudaStream_t stream);

// Host-side validation of blasst_decode's arguments other than the workspace
// (BLASST_OK or the status blasst_decode returns for them).
int decode_args_status(const void* q, const void* k_cache, const void* v_cache, const void* o, const float* lse,
                       int B, int Hq, int Hkv, int Lkv, int d, float scale, float lambda, int num_splits,
                       const unsigned long long* skipped_tiles_out, const float* margins);

}  // namespace blasst
