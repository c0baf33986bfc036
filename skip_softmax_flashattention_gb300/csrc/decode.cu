// decode.cu -- skip-softmax (BLASST) split-KV decode on sm_103a, plus the split merge.
//
// One CTA runs one (batch b, KV head hk, split s) pass over the split's key tiles
// in ascending order.  Its rows are the G = Hq/Hkv query heads that read KV head
// hk (one query token each), so one skip decision covers G rows x 128 keys and a
// V tile is loaded only when none of the G heads can skip it.
//
// The load order follows the BLASST decode design (BLASST talk notes, "kernel
// design: skip predicate reduction", Fig. 4): K tiles stream in ahead of use;
// each V tile is requested only after its tile's decision, so the HBM reads of
// skipped V tiles never happen.
//
// Both products run on the tensor cores with the key dimension on the 128 TMEM
// lanes:   S^T_j = K_j Q^T  (M = 128 keys, N = 16 padded heads, K = d)
//          O^T_j = V_j^T P_j^T (M = d = 128, N = 16, K = 128 keys)
// Each PV result lands in a fresh TMEM slot and is folded into per-thread
// registers (thread t owns output column t of every head) a few tiles later, so
// the decisions run ahead of the V loads and no TMEM read-modify-write is needed.
//
// Warp roles (224 threads): warps 0-3 softmax, warp 4 K loader, warp 5 MMA issuer
// and TMEM owner, warp 6 V loader.
//
// Head dim 64: the kernel runs at width 128.  The tensor maps have 64 columns, so the
// second 64-column box of every K and V tile lies outside the tensor and reads as
// zeros without touching memory; Q is staged with zero padding; only the first 64
// output columns are written.
//
// Paged form (blasst_decode_paged): K and V live in a pool of fixed-size pages and
// a page table maps each page-sized run of a sequence's keys to a physical page
// (The Hitchhiker's Guide, Phase 08, Section 3, "Paged Attention": key i of
// sequence b is row i mod page_size of page table[b][i / page_size]); every
// sequence has its own key count.  A 128-key
// tile is then fetched as 128 / page_size boxes (page_size < 128) or as one box
// inside a page (page_size a multiple of 128), through a 4-D tensor map over the
// pool.  Boxes past the end of the sequence, and boxes whose page index is out of
// range, get an out-of-range page coordinate: TMA writes zeros there and reads no
// memory (an out-of-range index is also reported in the device status word).
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace blasst {
namespace {

constexpr unsigned long long kDrainNs = 1000000000ull;

constexpr int D = 128;
constexpr int NPAD = 16;               // MMA N: the G heads padded to 16
constexpr int TILE_BYTES = kTile * D * 2;
constexpr int BOX_BYTES = kTile * 128;
constexpr int NK = 3, NV = 3;          // K / V shared-memory stages
constexpr int NS = 4, NO = 4;          // TMEM S / O slots (16 columns each)
constexpr int NP = 4;                  // P staging buffers
constexpr int ND = 8;                  // decision ring
constexpr int NH = 8;                  // reference-max history ring
constexpr int LOOKAHEAD = 3;           // S MMAs issued ahead of the PV MMA
constexpr int LAG = 2;                 // PV results folded this many computed tiles late
constexpr int Q_BYTES = (D / 64) * NPAD * 128;
constexpr int P_BYTES = 2 * NPAD * 128;  // [key half][16 rows][64 keys]
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + NK * TILE_BYTES;
constexpr int OFF_Q = OFF_V + NV * TILE_BYTES;
constexpr int OFF_P = OFF_Q + Q_BYTES;
constexpr int OFF_CTRL = OFF_P + NP * P_BYTES;
constexpr uint32_t TMEM_COLS = 128;
constexpr uint32_t O_COL = NS * NPAD;
static_assert(O_COL + NO * NPAD <= TMEM_COLS, "TMEM budget");
static_assert(LAG <= NO && LOOKAHEAD + 1 <= NS && LOOKAHEAD + 2 <= ND, "ring sizes");

struct DecodeCtrl {
    uint64_t k_full[NK], k_empty[NK], v_full[NV], v_empty[NV];
    uint64_t s_full[NS], s_free[NS], dec_full[ND], dec_free[ND];
    uint64_t p_full[NP], p_free[NP], o_full[NO], o_free[NO];
    uint64_t q_full, drain;
    uint32_t tmem_base;
    int dec[ND];
    int abort;
    float red[2][4][NPAD];
    float mref_hist[NH][NPAD];
    float lred[4][NPAD];
};
constexpr int SMEM = OFF_CTRL + (int)sizeof(DecodeCtrl) + 1024;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int G, bool PAGED>
__global__ void __launch_bounds__(224, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    DecodeCtrl* ctrl = reinterpret_cast<DecodeCtrl*>(smem + OFF_CTRL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    // This sequence's keys (its own count when seq_lens is given) and this split's
    // share of its tiles: split s takes tiles [s*nT/S, (s+1)*nT/S).
    int Lb = p.Lkv;
    if (p.seq_lens) {
        const int v = p.seq_lens[b];
        Lb = min(max(v, 0), p.Lkv);
        if (tid == 0 && s == 0 && hk == 0 && v != Lb) atomicOr(p.status, kStatusPageTable);
    }
    const int nTb = (Lb + kTile - 1) / kTile;
    // Sliding window: only keys [first_key, Lb); the splits share the tiles from the
    // one holding first_key.
    const int first_key = (p.window > 0 && Lb > p.window) ? Lb - p.window : 0;
    const int tlo = first_key / kTile;
    const int t0 = tlo + (int)(((long long)s * (nTb - tlo)) / p.S);
    const int t1 = tlo + (int)(((long long)(s + 1) * (nTb - tlo)) / p.S);
    const int n = t1 - t0;

    if (tid == 0) {
        for (int i = 0; i < NK; ++i) { mbar_init(&ctrl->k_full[i], 1); mbar_init(&ctrl->k_empty[i], 1); }
        for (int i = 0; i < NV; ++i) { mbar_init(&ctrl->v_full[i], 1); mbar_init(&ctrl->v_empty[i], 1); }
        for (int i = 0; i < NS; ++i) { mbar_init(&ctrl->s_full[i], 1); mbar_init(&ctrl->s_free[i], 4); }
        for (int i = 0; i < ND; ++i) {
            mbar_init(&ctrl->dec_full[i], 1);
            mbar_init(&ctrl->dec_free[i], 2);  // released by the MMA issuer and the V loader
        }
        for (int i = 0; i < NP; ++i) { mbar_init(&ctrl->p_full[i], 4); mbar_init(&ctrl->p_free[i], 1); }
        for (int i = 0; i < NO; ++i) { mbar_init(&ctrl->o_full[i], 1); mbar_init(&ctrl->o_free[i], 4); }
        mbar_init(&ctrl->q_full, 4);
        mbar_init(&ctrl->drain, 1);
        ctrl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(&ctrl->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    __syncwarp();  // the set-up above diverged inside warps; bar.sync is warp-aligned
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const Watchdog wd{&ctrl->abort, p.status, p.watchdog_ns};
    const int zkv = b * p.Hkv + hk;

    // Paged form: box i of a key tile covers its keys [i*rows, (i+1)*rows), one page
    // run; lane i of a loader warp reads that box's page index and issues it, so
    // the page-table reads of a tile are in flight together.
    const int nbox = PAGED ? kTile / p.rows_per_box : 1;
    // A page index is loaded ahead of its copy and checked only when the copy is issued
    // (a check right after the load would hold the loader warp for the whole load).
    auto box_live = [&](int tile, int i) -> bool {  // boxes past the keys or before the window read zeros
        const int key = tile * kTile + i * p.rows_per_box;
        return i < nbox && key < Lb && key + p.rows_per_box > first_key;
    };
    auto page_load = [&](int tile, int i) -> int {
        const int key = tile * kTile + i * p.rows_per_box;
        return box_live(tile, i) ? p.page_table[(long long)b * p.max_pages + key / p.page_size] : -1;
    };
    auto page_check = [&](int v, int tile, int i) -> int {
        if (!box_live(tile, i)) return p.num_pages;  // out of range: the box reads as zeros
        if (v >= 0 && v < p.num_pages) return v;
        atomicOr(p.status, kStatusPageTable);
        return p.num_pages;
    };
    // With up to kLane0Subs boxes a tile (pages of 32 keys or more) lane 0 issues them
    // all right after its slot wait, with page indices gathered once a tile; smaller
    // pages issue lane by lane after the wait's broadcast (a warp reconvergence then
    // sits between the freed slot and the copies).
    constexpr int kLane0Subs = 4;
    const bool lane0_issues = nbox <= kLane0Subs;
    auto issue_box = [&](const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int tile, int i, int pg) {
        const int off = (tile * kTile + i * p.rows_per_box) % p.page_size;
#pragma unroll
        for (int x = 0; x < D / 64; ++x) {
            uint8_t* dd = dst + x * BOX_BYTES + i * p.rows_per_box * 128;
            if (p.token_major)
                tma_load_4d(dd, map, bar, x * 64, hk, off, pg);
            else
                tma_load_4d(dd, map, bar, x * 64, off, hk, pg);
        }
    };

    if (warp == 4) {
        // ------------------------------------------------------------ K loader
        if constexpr (!PAGED) {
            if (lane == 0) {
                tma_prefetch_desc(&tk);
                int issued = 0;
                for (int j = 0; j < n; ++j) {
                    const int ks = j % NK;
                    if (j >= NK && !mbar_wait(&ctrl->k_empty[ks], ((j / NK) - 1) & 1, wd)) break;
                    mbar_arrive_expect_tx(&ctrl->k_full[ks], TILE_BYTES);
#pragma unroll
                    for (int x = 0; x < D / 64; ++x)
                        tma_load_3d(smem + OFF_K + ks * TILE_BYTES + x * BOX_BYTES, &tk, &ctrl->k_full[ks], x * 64,
                                    (t0 + j) * kTile, zkv);
                    issued = j + 1;
                }
                for (int j = max(0, issued - NK); j < issued; ++j)
                    mbar_wait_drain(&ctrl->k_full[j % NK], (j / NK) & 1, kDrainNs);
            }
        } else {
            if (lane == 0) tma_prefetch_desc(&tk);
            int issued = 0;
            // each lane's page index is read two tiles ahead of its copy
            int pg_next = n > 0 ? page_load(t0, lane) : 0;
            int pg_next2 = n > 1 ? page_load(t0 + 1, lane) : 0;
            for (int j = 0; j < n; ++j) {
                const int ks = j % NK;
                const int pg = page_check(pg_next, t0 + j, lane);
                int pgs[kLane0Subs];
#pragma unroll
                for (int i = 0; i < kLane0Subs; ++i) pgs[i] = __shfl_sync(0xffffffffu, pg, i);
                pg_next = pg_next2;
                pg_next2 = j + 2 < n ? page_load(t0 + j + 2, lane) : 0;
                int ok = 1;
                if (lane == 0) {
                    if (j >= NK && !mbar_wait(&ctrl->k_empty[ks], ((j / NK) - 1) & 1, wd)) {
                        ok = 0;
                    } else {
                        mbar_arrive_expect_tx(&ctrl->k_full[ks], TILE_BYTES);
                        if (lane0_issues) {
#pragma unroll
                            for (int i = 0; i < kLane0Subs; ++i)
                                if (i < nbox)
                                    issue_box(&tk, smem + OFF_K + ks * TILE_BYTES, &ctrl->k_full[ks], t0 + j, i, pgs[i]);
                        }
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                if (!lane0_issues && lane < nbox)
                    issue_box(&tk, smem + OFF_K + ks * TILE_BYTES, &ctrl->k_full[ks], t0 + j, lane, pg);
                issued = j + 1;
            }
            if (lane == 0)
                for (int j = max(0, issued - NK); j < issued; ++j)
                    mbar_wait_drain(&ctrl->k_full[j % NK], (j / NK) & 1, kDrainNs);
        }
    } else if (warp == 6) {
        // ------------------------------------------------------------ V loader
        if (lane == 0) tma_prefetch_desc(&tv);
        int comp = 0;
        int pg_next = (PAGED && n > 0) ? page_load(t0, lane) : 0;  // one tile ahead of its check
        for (int j = 0; j < n; ++j) {
            int pg = 0, pgs[kLane0Subs];
            if constexpr (PAGED) {
                pg = page_check(pg_next, t0 + j, lane);
#pragma unroll
                for (int i = 0; i < kLane0Subs; ++i) pgs[i] = __shfl_sync(0xffffffffu, pg, i);
                pg_next = j + 1 < n ? page_load(t0 + j + 1, lane) : 0;
            }
            const int vs = comp % NV;
            int go = 0;  // 0: stop, 1: load V_j, 2: tile skipped
            if (lane == 0) {
                if (mbar_wait(&ctrl->dec_full[j % ND], (j / ND) & 1, wd)) {
                    const bool skipped = reinterpret_cast<volatile int*>(ctrl->dec)[j % ND] != 0;
                    mbar_arrive(&ctrl->dec_free[j % ND]);
                    go = skipped ? 2 : 1;  // skipped: V never loaded
                    if (!skipped) {
                        if (comp >= NV && !mbar_wait(&ctrl->v_empty[vs], ((comp / NV) - 1) & 1, wd)) {
                            go = 0;
                        } else {
                            // the copies go out before the broadcast
                            mbar_arrive_expect_tx(&ctrl->v_full[vs], TILE_BYTES);
                            if constexpr (!PAGED) {
#pragma unroll
                                for (int x = 0; x < D / 64; ++x)
                                    tma_load_3d(smem + OFF_V + vs * TILE_BYTES + x * BOX_BYTES, &tv, &ctrl->v_full[vs],
                                                x * 64, (t0 + j) * kTile, zkv);
                            } else if (lane0_issues) {
#pragma unroll
                                for (int i = 0; i < kLane0Subs; ++i)
                                    if (i < nbox)
                                        issue_box(&tv, smem + OFF_V + vs * TILE_BYTES, &ctrl->v_full[vs], t0 + j, i,
                                                  pgs[i]);
                            }
                        }
                    }
                }
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            if (go == 0) break;
            if (go == 2) continue;
            if constexpr (PAGED) {
                if (!lane0_issues && lane < nbox)
                    issue_box(&tv, smem + OFF_V + vs * TILE_BYTES, &ctrl->v_full[vs], t0 + j, lane, pg);
            }
            ++comp;
        }
        if (lane == 0)
            for (int c = max(0, comp - NV); c < comp; ++c)
                mbar_wait_drain(&ctrl->v_full[c % NV], (c / NV) & 1, kDrainNs);
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16(128, NPAD, false, false);
            constexpr uint32_t kIdescO = idesc_bf16(D, NPAD, true, false);
            const uint32_t sK = smem_u32(smem + OFF_K), sV = smem_u32(smem + OFF_V);
            const uint32_t sQ = smem_u32(smem + OFF_Q), sP = smem_u32(smem + OFF_P);
            auto issue_s = [&](int j) -> bool {
                const int ks = j % NK, ss = j % NS;
                if (!mbar_wait(&ctrl->k_full[ks], (j / NK) & 1, wd)) return false;
                if (j >= NS && !mbar_wait(&ctrl->s_free[ss], ((j / NS) - 1) & 1, wd)) return false;
                tc_fence_after();
                const uint32_t kb = sK + ks * TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ao = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
                    const uint32_t bo = (kk >> 2) * (NPAD * 128) + (kk & 3) * 32;
                    mma_ss(tmem + ss * NPAD, desc_kmajor_sw128(kb + ao), desc_kmajor_sw128(sQ + bo), kIdescS,
                           kk > 0 ? 1u : 0u);
                }
                mma_commit(&ctrl->s_full[ss]);
                mma_commit(&ctrl->k_empty[ks]);
                return true;
            };
            bool ok = mbar_wait(&ctrl->q_full, 0, wd);
            for (int j = 0; j < min(LOOKAHEAD, n) && ok; ++j) ok = issue_s(j);
            int comp = 0;
            for (int j = 0; j < n && ok; ++j) {
                if (j + LOOKAHEAD < n && !(ok = issue_s(j + LOOKAHEAD))) break;
                if (!(ok = mbar_wait(&ctrl->dec_full[j % ND], (j / ND) & 1, wd))) break;
                const bool skipped = reinterpret_cast<volatile int*>(ctrl->dec)[j % ND] != 0;
                mbar_arrive(&ctrl->dec_free[j % ND]);
                if (skipped) continue;
                const int pb = comp % NP, vs = comp % NV, os = comp % NO;
                if (!(ok = mbar_wait(&ctrl->p_full[pb], (comp / NP) & 1, wd))) break;
                if (!(ok = mbar_wait(&ctrl->v_full[vs], (comp / NV) & 1, wd))) break;
                if (comp >= NO && !(ok = mbar_wait(&ctrl->o_free[os], ((comp / NO) - 1) & 1, wd))) break;
                tc_fence_after();
                const uint32_t vb = sV + vs * TILE_BYTES, pbuf = sP + pb * P_BYTES;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    const uint64_t adesc = desc_mnmajor_sw128(vb + kk * 2048, BOX_BYTES);
                    const uint64_t bdesc = desc_kmajor_sw128(pbuf + (kk >> 2) * (NPAD * 128) + (kk & 3) * 32);
                    mma_ss(tmem + O_COL + os * NPAD, adesc, bdesc, kIdescO, kk > 0 ? 1u : 0u);
                }
                mma_commit(&ctrl->o_full[os]);
                mma_commit(&ctrl->v_empty[vs]);
                mma_commit(&ctrl->p_free[pb]);
                ++comp;
            }
            mma_commit(&ctrl->drain);
            mbar_wait_drain(&ctrl->drain, 0, kDrainNs);
        }
    } else {
        // ------------------------------------------------------------ softmax (warps 0-3)
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        // Stage Q (rows = heads, zero-padded to 16) and clear the P buffers' padding rows.
        {
            uint8_t* sq = smem + OFF_Q;
            for (int c = tid; c < NPAD * (D / 8); c += 128) {
                const int g = c / (D / 8), ck = c % (D / 8);
                uint4 v = make_uint4(0, 0, 0, 0);
                if (g < G && ck * 8 < p.d)
                    v = *reinterpret_cast<const uint4*>(p.q + ((long long)b * p.Hq + hk * G + g) * p.d + ck * 8);
                const int half = ck >> 3, cw = ck & 7;
                *reinterpret_cast<uint4*>(sq + half * (NPAD * 128) + g * 128 + ((cw ^ (g & 7)) << 4)) = v;
            }
            uint4* sp = reinterpret_cast<uint4*>(smem + OFF_P);
            for (int c = tid; c < NP * P_BYTES / 16; c += 128) sp[c] = make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctrl->q_full);
        }
        const long long mapbase = (long long)zkv * p.nK;
        const float cl = p.c_log2;
        float m_exact[G], m_ref[G], lpart[G], oacc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m_exact[g] = -CUDART_INF_F;
            m_ref[g] = -CUDART_INF_F;
            lpart[g] = 0.f;
            oacc[g] = 0.f;
        }
        int comp = 0, folded = 0;
        unsigned long long nskip = 0;

        auto fold = [&](int i) {
            const int os = i % NO;
            mbar_wait(&ctrl->o_full[os], (i / NO) & 1, wd);
            tc_fence_after();
            uint32_t yr[16];
            tmem_ld16(tl + O_COL + os * NPAD, yr);
            tmem_ld_wait();
            fence_regs<16>(yr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctrl->o_free[os]);
            const volatile float* mh = ctrl->mref_hist[i % NH];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float f = (mh[g] == m_ref[g]) ? 1.f : ex2((mh[g] - m_ref[g]) * cl);
                oacc[g] = fmaf(f, __uint_as_float(yr[g]), oacc[g]);
            }
        };

        for (int j = 0; j < n; ++j) {
            const int ss = j % NS;
            mbar_wait(&ctrl->s_full[ss], (j / NS) & 1, wd);
            tc_fence_after();
            uint32_t xr[16];
            tmem_ld16(tl + ss * NPAD, xr);
            tmem_ld_wait();
            fence_regs<16>(xr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctrl->s_free[ss]);
            const int key = (t0 + j) * kTile + tid;
            const bool key_ok = key < Lb && key >= first_key;
            float x[G];
#pragma unroll
            for (int g = 0; g < G; ++g) x[g] = key_ok ? __uint_as_float(xr[g]) : -CUDART_INF_F;
            // per-head tile max over the 128 keys: warp shuffle, then across the 4 warps
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float v = x[g];
#pragma unroll
                for (int sh = 16; sh > 0; sh >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, sh));
                if (lane == 0) ctrl->red[j & 1][warp][g] = v;
            }
            named_bar_sync(1, 128);
            float mnew[G];
            bool skip = true;
            float margin = -CUDART_INF_F;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const volatile float* rd = &ctrl->red[j & 1][0][g];
                const float mt = fmaxf(fmaxf(rd[0], rd[NPAD]), fmaxf(rd[2 * NPAD], rd[3 * NPAD]));
                mnew[g] = fmaxf(m_exact[g], mt);
                const float diff = mt - mnew[g];
                skip = skip && (diff < p.thr_raw);
                const float gm = (mt == -CUDART_INF_F && mnew[g] == -CUDART_INF_F) ? CUDART_INF_F : diff;
                margin = fmaxf(margin, gm);
                m_exact[g] = mnew[g];
            }
            if (tid == 0) {
                // the slot is reused only after both readers of tile j - ND released it
                if (j >= ND) mbar_wait(&ctrl->dec_free[j % ND], ((j / ND) - 1) & 1, wd);
                reinterpret_cast<volatile int*>(ctrl->dec)[j % ND] = skip ? 1 : 0;
                mbar_arrive(&ctrl->dec_full[j % ND]);
                if (p.skip_map) p.skip_map[mapbase + t0 + j] = skip ? 1 : 0;
                if (p.margins) p.margins[mapbase + t0 + j] = margin * p.scale;
                nskip += skip ? 1 : 0;
            }
            if (!skip) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (mnew[g] != -CUDART_INF_F && (m_ref[g] == -CUDART_INF_F || mnew[g] > m_ref[g] + p.lazy_raw)) {
                        const float a = m_ref[g] == -CUDART_INF_F ? 0.f : ex2((m_ref[g] - mnew[g]) * cl);
                        oacc[g] *= a;
                        lpart[g] *= a;
                        m_ref[g] = mnew[g];
                    }
                }
                if (tid == 0) {
#pragma unroll
                    for (int g = 0; g < G; ++g) ctrl->mref_hist[comp % NH][g] = m_ref[g];
                }
                const int pb = comp % NP;
                if (comp >= NP) mbar_wait(&ctrl->p_free[pb], ((comp / NP) - 1) & 1, wd);
                uint8_t* pbuf = smem + OFF_P + pb * P_BYTES + (tid >> 6) * (NPAD * 128);
                const int cw = (tid & 63) >> 3;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float mr = m_ref[g] == -CUDART_INF_F ? 0.f : m_ref[g];
                    const float pv = ex2(fmaf(x[g], cl, -mr * cl));
                    lpart[g] += pv;
                    *reinterpret_cast<unsigned short*>(pbuf + g * 128 + ((cw ^ (g & 7)) << 4) + (tid & 7) * 2) =
                        (unsigned short)(pack_bf16x2(pv, 0.f) & 0xffffu);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctrl->p_full[pb]);
                ++comp;
            }
            while (comp - folded > LAG) fold(folded++);
        }
        named_bar_sync(1, 128);
        while (folded < comp) fold(folded++);

        // l = sum over the 128 key lanes; O = oacc / l
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float v = lpart[g];
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) v += __shfl_xor_sync(0xffffffffu, v, sh);
            if (lane == 0) ctrl->lred[warp][g] = v;
        }
        named_bar_sync(1, 128);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const volatile float* lr = &ctrl->lred[0][g];
            const float l = lr[0] + lr[NPAD] + lr[2 * NPAD] + lr[3 * NPAD];
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const float lse = l > 0.f ? m_ref[g] * p.scale + __logf(l) : -CUDART_INF_F;
            const long long hq = (long long)b * p.Hq + hk * G + g;
            if (p.S == 1) {
                if (tid < p.d)
                    reinterpret_cast<unsigned short*>(p.o)[hq * p.d + tid] =
                        (unsigned short)(pack_bf16x2(oacc[g] * inv, 0.f) & 0xffffu);
                if (tid == 0 && p.lse) p.lse[hq] = lse;
            } else {
                const long long ps = (long long)s * p.B * p.Hq + hq;
                if (tid < p.d) p.o_part[ps * p.d + tid] = oacc[g] * inv;
                if (tid == 0) p.lse_part[ps] = lse;
            }
        }
        if (tid == 0 && p.skipped && nskip) atomicAdd(p.skipped, nskip);
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Merge the per-split results by log-sum-exp: lse = ln(sum_s e^{lse_s}),
// O = sum_s e^{lse_s - lse} O_s.  One CTA per (head, batch), one thread per column.
// Each warp reads the split lse values lane by lane (split s in lane s mod 32) and
// reduces their max and sum with shuffles, so the reads are in flight together; the
// weighted sum then streams the partials with independent loads.  (Reading the lse
// values split after split in every thread made the merge latency-bound: 12.8 us for
// 7 splits of 64 x 16 rows of 512 values.)
__global__ void combine_kernel(const CombineParams p) {
    const int hq = blockIdx.x, b = blockIdx.y, t = threadIdx.x, lane = t & 31;
    const long long bh = (long long)b * p.Hq + hq;
    const long long stride = (long long)p.B * p.Hq;
    float M = -CUDART_INF_F;
    for (int s = lane; s < p.S; s += 32) M = fmaxf(M, p.lse_part[s * stride + bh]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M == -CUDART_INF_F) {  // no split saw a key (a sequence of length 0)
        reinterpret_cast<unsigned short*>(p.o)[bh * p.d + t] = 0;
        if (t == 0 && p.lse) p.lse[bh] = -CUDART_INF_F;
        return;
    }
    float tot = 0.f;
    for (int s = lane; s < p.S; s += 32) tot += __expf(p.lse_part[s * stride + bh] - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    const float L = M + __logf(tot);
    float acc = 0.f;
#pragma unroll 4
    for (int s = 0; s < p.S; ++s) {
        const float w = __expf(p.lse_part[s * stride + bh] - L);
        acc = fmaf(w, p.o_part[(s * stride + bh) * p.d + t], acc);
    }
    reinterpret_cast<unsigned short*>(p.o)[bh * p.d + t] = (unsigned short)(pack_bf16x2(acc, 0.f) & 0xffffu);
    if (t == 0 && p.lse) p.lse[bh] = L;
}

template <int G, bool PAGED>
cudaError_t launch_gp(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<G, PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(p.S, p.Hkv, p.B);
    decode_kernel<G, PAGED><<<grid, 224, SMEM, stream>>>(tk, tv, p);
    return cudaGetLastError();
}
template <int G>
cudaError_t launch_g(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, cudaStream_t stream) {
    return p.page_table ? launch_gp<G, true>(tk, tv, p, stream) : launch_gp<G, false>(tk, tv, p, stream);
}

}  // namespace

cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, int d,
                          cudaStream_t stream) {
    (void)d;
    switch (p.G) {
        case 1: return launch_g<1>(tk, tv, p, stream);
        case 2: return launch_g<2>(tk, tv, p, stream);
        case 4: return launch_g<4>(tk, tv, p, stream);
        case 8: return launch_g<8>(tk, tv, p, stream);
        case 16: return launch_g<16>(tk, tv, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    dim3 grid(p.Hq, p.B);
    combine_kernel<<<grid, p.d, 0, stream>>>(p);
    return cudaGetLastError();
}

size_t decode_smem_bytes(int d) {
    (void)d;
    return SMEM;
}

}  // namespace blasst
