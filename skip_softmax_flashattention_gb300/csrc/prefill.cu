// prefill.cu -- skip-softmax (BLASST) FlashAttention forward for prefill on sm_103a.
//
// Two kernels: prefill2_kernel, the default, runs two query tiles per CTA with their
// softmaxes half a period apart on the tensor core (described where it is defined);
// prefill_kernel, described here, runs one query tile per CTA and serves the
// BLASST_PREFILL_ONE_QTILE and BLASST_PREFILL_P_VIA_SMEM variants.
//
// One CTA computes one 128-row query tile of one query head against the key tiles
// it can see, in ascending order (Hitchhiker's Guide Phase 08, Section 1,
// "FlashAttention Tiling Strategy"), with the BLASST per-tile test between S and
// the softmax (Skip-Softmax design doc, "Algorithm"; BLASST talk notes, Eq. 2).
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t = TMEM lane t.  Reads S_j from
//              TMEM, masks, takes the row's tile max m~, updates the exact running
//              max m, votes (m~ - m < ln lambda), reduces the vote with __all and a
//              shared-memory atomicAnd across the four warps (BLASST talk notes,
//              "kernel design: skip predicate reduction"), and for computed tiles
//              writes P = 2^(S*c - m_ref*c) (bf16) and rescales its O row when the
//              reference max moves.
//   warp 4     TMA producer: Q once, then K_j / V_j into a ring of shared-memory
//              stages (128-byte swizzled boxes of 64 columns).
//   warp 5     MMA issuer (one thread) and TMEM owner: S_j = Q K_j^T into one of
//              two TMEM S buffers (issued one tile ahead so the tensor core runs
//              while the softmax works), and O += P_j V_j for computed tiles only.
//
// Skipped tiles omit the exponentials, the row sums and the P.V product; the V
// tile is still staged (the prefill kernel keeps its prefetch predictable, as the
// BLASST kernel design describes for prefill).
//
// TMEM columns: S buffer 0 = [0,128), S buffer 1 = [128,256), O = [256, 256+D).
// When P lives in TMEM it overwrites the first 64 columns of its S buffer (two
// bf16 per 32-bit column); otherwise it is staged in shared memory.
//
// The reference max m_ref used for the exponentials only moves when the exact
// running max exceeds it by more than `lazy_raw` (2^8 in probability units), so
// the O rescale (a TMEM read-modify-write) is rare; the skip test always uses the
// exact running max.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "kernels.cuh"
#include "ptx.cuh"


namespace blasst {
namespace {

constexpr unsigned long long kDrainNs = 1000000000ull;  // drain waits: 1 s

template <int NK, int NV>
struct PrefillCtrl {
    uint64_t q_full;
    uint64_t k_full[NK], k_empty[NK];
    uint64_t v_full[NV], v_empty[NV];
    uint64_t s_full[2], p_full[2], p_free[2];
    uint64_t o_done, drain, never;
    uint32_t tmem_base;
    int vote[3];
    int dec[2];
    int abort;
    float mred[2][4];
};

template <int D, bool PT>
struct PrefillCfg {
    static constexpr int TILE_BYTES = kTile * D * 2;  // a 128 x D bf16 tile
    static constexpr int BOX_BYTES = kTile * 128;     // one 128-row box of 64 bf16 columns
    static constexpr int NK = (D == 128) ? (PT ? 3 : 2) : (PT ? 4 : 3);
    static constexpr int NV = NK;
    static constexpr int P_BYTES = PT ? 0 : 2 * kTile * kTile * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NK * TILE_BYTES;
    static constexpr int OFF_P = OFF_V + NV * TILE_BYTES;
    static constexpr int OFF_CTRL = OFF_P + P_BYTES;
    using Ctrl = PrefillCtrl<NK, NV>;
    static constexpr int SMEM = OFF_CTRL + (int)sizeof(Ctrl) + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t O_COL = 256;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D, bool PT>
__global__ void __launch_bounds__(192, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const PrefillParams p) {
    using C = PrefillCfg<D, PT>;
    using Ctrl = typename C::Ctrl;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + C::OFF_CTRL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int G = p.Hq / p.Hkv;
    int unit, b, h;
    prefill_cta_coords(p, p.nQ, unit, b, h);
    const int qt = p.causal ? (p.nQ - 1 - unit) : unit;  // heavy tiles first
    const int hk = h / G;
    const int r0 = qt * kTile;
    const int rows = min(kTile, p.Lq - r0);
    const int off = p.Lkv - p.Lq;  // bottom-right causal alignment
    int n = p.nK;                  // key tiles visited
    if (p.causal) {
        const int maxkey = r0 + rows - 1 + off;
        n = maxkey < 0 ? 0 : min(p.nK, maxkey / kTile + 1);
    }

    if (tid == 0) {
        mbar_init(&ctrl->q_full, 1);
        for (int i = 0; i < C::NK; ++i) {
            mbar_init(&ctrl->k_full[i], 1);
            mbar_init(&ctrl->k_empty[i], 1);
        }
        for (int i = 0; i < C::NV; ++i) {
            mbar_init(&ctrl->v_full[i], 1);
            mbar_init(&ctrl->v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctrl->s_full[i], 1);
            mbar_init(&ctrl->p_full[i], 4);
            mbar_init(&ctrl->p_free[i], 1);
        }
        mbar_init(&ctrl->o_done, 1);
        mbar_init(&ctrl->drain, 1);
        mbar_init(&ctrl->never, 1);
        ctrl->vote[0] = ctrl->vote[1] = ctrl->vote[2] = 1;
        ctrl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(&ctrl->tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    __syncwarp();  // the set-up above diverged inside warps; bar.sync is warp-aligned
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const Watchdog wd{&ctrl->abort, p.status, p.watchdog_ns};

    if (warp == 4) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            const int zq = b * p.Hq + h, zkv = b * p.Hkv + hk;
            mbar_arrive_expect_tx(&ctrl->q_full, C::TILE_BYTES);
#pragma unroll
            for (int x = 0; x < D / 64; ++x)
                tma_load_3d(smem + C::OFF_Q + x * C::BOX_BYTES, &tq, &ctrl->q_full, x * 64, r0, zq);
            int issued_k = 0, issued_v = 0;
            for (int j = 0; j < n; ++j) {
                const int ks = j % C::NK;
                if (j >= C::NK && !mbar_wait(&ctrl->k_empty[ks], ((j / C::NK) - 1) & 1, wd)) break;
                mbar_arrive_expect_tx(&ctrl->k_full[ks], C::TILE_BYTES);
#pragma unroll
                for (int x = 0; x < D / 64; ++x)
                    tma_load_3d(smem + C::OFF_K + ks * C::TILE_BYTES + x * C::BOX_BYTES, &tk, &ctrl->k_full[ks],
                                x * 64, j * kTile, zkv);
                issued_k = j + 1;
                const int vs = j % C::NV;
                if (j >= C::NV && !mbar_wait(&ctrl->v_empty[vs], ((j / C::NV) - 1) & 1, wd)) break;
                mbar_arrive_expect_tx(&ctrl->v_full[vs], C::TILE_BYTES);
#pragma unroll
                for (int x = 0; x < D / 64; ++x)
                    tma_load_3d(smem + C::OFF_V + vs * C::TILE_BYTES + x * C::BOX_BYTES, &tv, &ctrl->v_full[vs],
                                x * 64, j * kTile, zkv);
                issued_v = j + 1;
            }
            // Every copy this thread started must land before the CTA can exit.
            mbar_wait_drain(&ctrl->q_full, 0, kDrainNs);
            for (int j = max(0, issued_k - C::NK); j < issued_k; ++j)
                mbar_wait_drain(&ctrl->k_full[j % C::NK], (j / C::NK) & 1, kDrainNs);
            for (int j = max(0, issued_v - C::NV); j < issued_v; ++j)
                mbar_wait_drain(&ctrl->v_full[j % C::NV], (j / C::NV) & 1, kDrainNs);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n > 0) {
            constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
            constexpr uint32_t kIdescO = idesc_bf16(128, D, false, true);
            const uint32_t sQ = smem_u32(smem + C::OFF_Q);
            const uint32_t sK = smem_u32(smem + C::OFF_K);
            const uint32_t sV = smem_u32(smem + C::OFF_V);
            const uint32_t sP = smem_u32(smem + C::OFF_P);
            auto issue_s = [&](int j) -> bool {
                const int ks = j % C::NK;
                if (!mbar_wait(&ctrl->k_full[ks], (j / C::NK) & 1, wd)) return false;
                tc_fence_after();
                const uint32_t dcol = tmem + (uint32_t)(j & 1) * 128u;
                const uint32_t kb = sK + ks * C::TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t o = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
                    mma_ss(dcol, desc_kmajor_sw128(sQ + o), desc_kmajor_sw128(kb + o), kIdescS, kk > 0 ? 1u : 0u);
                }
                mma_commit(&ctrl->s_full[j & 1]);
                mma_commit(&ctrl->k_empty[ks]);
                return true;
            };
            // test hook: a wait on a barrier nothing arrives on runs into the watchdog
            bool ok = p.test_stall ? mbar_wait(&ctrl->never, 0, wd) : true;
            ok = ok && mbar_wait(&ctrl->q_full, 0, wd);
            if (ok) ok = issue_s(0);
            int npv = 0;
            for (int j = 0; j < n && ok; ++j) {
                if (j + 1 < n && !(ok = issue_s(j + 1))) break;
                if (!(ok = mbar_wait(&ctrl->p_full[j & 1], (j >> 1) & 1, wd))) break;
                const int vs = j % C::NV;
                if (!(ok = mbar_wait(&ctrl->v_full[vs], (j / C::NV) & 1, wd))) break;
                tc_fence_after();
                const bool skip = reinterpret_cast<volatile int*>(ctrl->dec)[j & 1] != 0;
                if (!skip) {
                    const uint32_t vb = sV + vs * C::TILE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk) {
                        const uint64_t bdesc = desc_mnmajor_sw128(vb + kk * 2048, C::BOX_BYTES);
                        const uint32_t acc = (npv > 0 || kk > 0) ? 1u : 0u;
                        if constexpr (PT) {
                            mma_ts(tmem + C::O_COL, tmem + (uint32_t)(j & 1) * 128u + kk * 8, bdesc, kIdescO, acc);
                        } else {
                            const uint32_t pa = sP + (j & 1) * (kTile * kTile * 2) + (kk >> 2) * C::BOX_BYTES +
                                                (kk & 3) * 32;
                            mma_ss(tmem + C::O_COL, desc_kmajor_sw128(pa), bdesc, kIdescO, acc);
                        }
                    }
                    mma_commit(&ctrl->o_done);
                    if constexpr (!PT) mma_commit(&ctrl->p_free[j & 1]);
                    mma_commit(&ctrl->v_empty[vs]);
                    ++npv;
                } else {
                    mbar_arrive(&ctrl->v_empty[vs]);
                }
            }
            mma_commit(&ctrl->drain);
            mbar_wait_drain(&ctrl->drain, 0, kDrainNs);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int row = tid;
        const int rabs = r0 + row;
        const bool valid = rabs < p.Lq;
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        const int lim_row = p.causal ? rabs + off : 0x3fffffff;
        const long long mapbase = ((long long)(b * p.Hq + h) * p.nQ + qt) * p.nK;
        float m_exact = -CUDART_INF_F, m_ref = -CUDART_INF_F, l = 0.f;
        int npv = 0;
        int puse0 = 0, puse1 = 0;
        unsigned long long nskip = 0;
        uint8_t* sP = smem + C::OFF_P;

        for (int j = 0; j < n; ++j) {
            mbar_wait(&ctrl->s_full[j & 1], (j >> 1) & 1, wd);
            tc_fence_after();
            uint32_t xr[128];
            float lm[4];  // maximum of each 32-column quarter (load and reduce)
            const uint32_t sc = tl + (uint32_t)(j & 1) * 128u;
            tmem_ld32_max(sc + 0, xr, lm[0]);
            tmem_ld32_max(sc + 32, xr + 32, lm[1]);
            tmem_ld32_max(sc + 64, xr + 64, lm[2]);
            tmem_ld32_max(sc + 96, xr + 96, lm[3]);
            tmem_ld_wait();
            fence_regs<128>(xr);
            asm volatile("" : "+f"(lm[0]), "+f"(lm[1]), "+f"(lm[2]), "+f"(lm[3]));  // used after the wait

            // mask keys beyond Lkv and (causal) beyond the row's diagonal
            const int lim = min(p.Lkv - 1, lim_row) - j * kTile;
            float mt = fmaxf(fmaxf(lm[0], lm[1]), fmaxf(lm[2], lm[3]));
            if (lim < kTile - 1) {
#pragma unroll
                for (int c = 0; c < kTile; ++c)
                    if (c > lim) xr[c] = __float_as_uint(-CUDART_INF_F);
                mt = row_max128(xr);
            }
            const float mnew = fmaxf(m_exact, mt);
            const float diff = mt - mnew;  // NaN when both are -inf: votes "compute"
            const bool vote = !valid || (diff < p.thr_raw);
            const unsigned all = __all_sync(0xffffffffu, vote);
            if (lane == 0) atomicAnd(&ctrl->vote[j % 3], (int)all);
            if (p.margins) {
                float g = valid ? ((mt == -CUDART_INF_F && mnew == -CUDART_INF_F) ? CUDART_INF_F : diff)
                                : -CUDART_INF_F;
#pragma unroll
                for (int s = 16; s > 0; s >>= 1) g = fmaxf(g, __shfl_xor_sync(0xffffffffu, g, s));
                if (lane == 0) ctrl->mred[j & 1][warp] = g;
            }
            named_bar_sync(1, 128);
            const bool skip = reinterpret_cast<volatile int*>(ctrl->vote)[j % 3] != 0;
            if (tid == 0) {
                ctrl->vote[(j + 2) % 3] = 1;
                reinterpret_cast<volatile int*>(ctrl->dec)[j & 1] = skip ? 1 : 0;
                if (p.skip_map) p.skip_map[mapbase + j] = skip ? 1 : 0;
                if (p.margins) {
                    const volatile float* mr = ctrl->mred[j & 1];
                    const float g = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3]));
                    p.margins[mapbase + j] = g * p.scale;
                }
                nskip += skip ? 1 : 0;
            }
            m_exact = mnew;

            if (!skip) {
                // move the reference max (rarely, see lazy_raw) and rescale this row of O
                const bool move = mnew != -CUDART_INF_F && (m_ref == -CUDART_INF_F || mnew > m_ref + p.lazy_raw);
                const float alpha = move ? (m_ref == -CUDART_INF_F ? 0.f : ex2((m_ref - mnew) * p.c_log2)) : 1.f;
                if (__any_sync(0xffffffffu, move) && npv > 0) {
                    mbar_wait(&ctrl->o_done, (npv - 1) & 1, wd);
                    tc_fence_after();
#pragma unroll
                    for (int cc = 0; cc < D; cc += 32) {
                        uint32_t t[32];
                        tmem_ld32(tl + C::O_COL + cc, t);
                        tmem_ld_wait();
                        fence_regs<32>(t);
#pragma unroll
                        for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
                        tmem_st32(tl + C::O_COL + cc, t);
                    }
                    tmem_st_wait();
                }
                if (move) {
                    l *= alpha;
                    m_ref = mnew;
                }
                const float mc = (m_ref == -CUDART_INF_F ? 0.f : m_ref) * p.c_log2;
                const float cl = p.c_log2;
                if constexpr (!PT) {
                    const int pb = j & 1;
                    const int uses = pb ? puse1 : puse0;
                    if (uses > 0) mbar_wait(&ctrl->p_free[pb], (uses - 1) & 1, wd);
                }
                float rs = 0.f;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float p0 = ex2(fmaf(__uint_as_float(xr[ch * 32 + 2 * i]), cl, -mc));
                        const float p1 = ex2(fmaf(__uint_as_float(xr[ch * 32 + 2 * i + 1]), cl, -mc));
                        rs += p0 + p1;
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    if constexpr (PT) {
                        tmem_st16(tl + (uint32_t)(j & 1) * 128u + ch * 16, pk);
                    } else {
                        // P buffer: [key half][128 rows][64 keys], 16-byte chunks swizzled by row
                        uint8_t* pbuf = sP + (j & 1) * (kTile * kTile * 2) + (ch >> 1) * C::BOX_BYTES + row * 128;
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const int chunk = (ch & 1) * 4 + q4;
                            uint4 v4 = make_uint4(pk[q4 * 4], pk[q4 * 4 + 1], pk[q4 * 4 + 2], pk[q4 * 4 + 3]);
                            *reinterpret_cast<uint4*>(pbuf + ((chunk ^ (row & 7)) << 4)) = v4;
                        }
                    }
                }
                l += rs;
                ++npv;
                if constexpr (PT) {
                    tmem_st_wait();
                } else {
                    if (j & 1) ++puse1; else ++puse0;
                    fence_proxy_async_smem();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctrl->p_full[j & 1]);
        }

        // ---------------------------------------------------------------- epilogue
        if (npv > 0) {
            mbar_wait(&ctrl->o_done, (npv - 1) & 1, wd);
            tc_fence_after();
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + ((long long)(b * p.Hq + h) * p.Lq + rabs) * D;
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
            uint32_t t[32];
            if (npv > 0) {
                tmem_ld32(tl + C::O_COL + cc, t);
                tmem_ld_wait();
                fence_regs<32>(t);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) t[i] = 0u;
            }
            if (valid) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 v4;
                    v4.x = pack_bf16x2(__uint_as_float(t[q4 * 8 + 0]) * inv, __uint_as_float(t[q4 * 8 + 1]) * inv);
                    v4.y = pack_bf16x2(__uint_as_float(t[q4 * 8 + 2]) * inv, __uint_as_float(t[q4 * 8 + 3]) * inv);
                    v4.z = pack_bf16x2(__uint_as_float(t[q4 * 8 + 4]) * inv, __uint_as_float(t[q4 * 8 + 5]) * inv);
                    v4.w = pack_bf16x2(__uint_as_float(t[q4 * 8 + 6]) * inv, __uint_as_float(t[q4 * 8 + 7]) * inv);
                    *reinterpret_cast<uint4*>(orow + cc + q4 * 8) = v4;
                }
            }
        }
        if (valid && p.lse) {
            p.lse[(long long)(b * p.Hq + h) * p.Lq + rabs] =
                l > 0.f ? m_ref * p.scale + __logf(l) : -CUDART_INF_F;
        }
        if (tid == 0 && p.skipped && nskip) atomicAdd(p.skipped, nskip);
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ============================================================================
// Two query tiles per CTA (the default path).
//
// The CTA owns query tiles A = 2i and B = 2i+1 of one head; each K/V tile is
// staged once and used by both.  Warps 0-3 run the softmax of tile A, warps 4-7
// that of tile B, warp 8 loads Q and the K tiles, warp 11 the V tiles, warps 9 and
// 10 issue the MMAs of tiles A and B (one thread each, so that one issuer's barrier
// waits overlap the other's MMAs).  Registers: 168 per thread at launch, 72 for
// warpgroup 2 and 216 for the softmax warpgroups afterwards -- 2*128*216 + 128*72 =
// 384*168.  TMEM:
// S_A = [0,128), S_B = [128,256), O_A = [256, 256+D), O_B = [256+D, 256+2D);
// P_w overwrites the first 64 columns of S_w.  The tensor core runs, per key
// tile j:  ... PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1) ...  so the softmax of one
// tile runs while the tensor core works on the other tile.  The tensor core queues
// only a couple of MMAs ahead, so every instruction the issuing thread spends
// between MMAs (a barrier wait, a commit) can leave it idle: each issuer commits
// once per key tile, and that one commit tells the softmax that S is ready and
// the producer which K/V slots its tile has finished with (a commit arrives only
// after all earlier MMAs of its thread).  The producer waits only for the issuers
// whose tile read the previous occupant of a slot.
// ============================================================================
template <int NK, int NV>
struct Prefill2Ctrl {
    // Commit c of the MMA issuer of query tile w arrives on rel[w][c % NR] once QK_w(c)
    // and PV_w(c-1) -- and every MMA that thread issued before them -- are done: the
    // softmax waits commit j for S_j (and for O to hold PV_w(j-1) before a rescale), the
    // producer waits it to reuse K and V slots.  NR > max(NK, NV) keeps every waiter
    // within one phase of the barrier it waits on.
    static constexpr int NR = (NK > NV ? NK : NV) + 1;
    uint64_t q_full;
    uint64_t k_full[NK], v_full[NV];
    uint64_t rel[2][NR];
    uint64_t p_full[2][2];  // p_full[w][0]: tile w voted (and stored P's first half, keys 0..63,
                            // on a computed tile); p_full[w][1]: P's second half (computed tiles only)
    uint64_t never;
    uint32_t tmem_base;
    int keep[2];  // keep[w] = j+1 once a warp of tile w keeps key tile j (only grows)
    int dec[2];   // V elision: 2(j+1) + kept, tile w's decision on key tile j, from its issuer (only grows)
    int v_issued; // V tiles the V producer has issued (or completed without data); only grows
    int abort;
    int turn;       // which issuer may put its next group of MMAs into the tensor queue
    int active[2];  // issuer w still has key tiles to process
    float mred[2][2][4];
};

template <int D>
struct Prefill2Cfg {
    static constexpr int TILE_BYTES = kTile * D * 2;
    static constexpr int BOX_BYTES = kTile * 128;
    static constexpr int NK = (D == 128) ? 3 : 4;
    static constexpr int NV = (D == 128) ? 2 : 4;
    static constexpr int OFF_Q = 0;  // Q_A, then Q_B
    static constexpr int OFF_K = 2 * TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NK * TILE_BYTES;
    static constexpr int OFF_CTRL = OFF_V + NV * TILE_BYTES;
    using Ctrl = Prefill2Ctrl<NK, NV>;
    static constexpr int SMEM = OFF_CTRL + (int)sizeof(Ctrl) + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t O_COL = 256;
};

constexpr int kRegsLaunch2 = 168, kRegsSoftmax2 = 216, kRegsProducer2 = 72;
static_assert(2 * 128 * kRegsSoftmax2 + 128 * kRegsProducer2 <= 384 * kRegsLaunch2, "register split");

template <int D, bool WIN>
__global__ void __launch_bounds__(384, 1)
    prefill2_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const PrefillParams p) {
    using C = Prefill2Cfg<D>;
    using Ctrl = typename C::Ctrl;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + C::OFF_CTRL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int G = p.Hq / p.Hkv;
    const int npairs = (p.nQ + 1) >> 1;
    int unit, b, h;
    prefill_cta_coords(p, npairs, unit, b, h);
    const int pi = p.causal ? (npairs - 1 - unit) : unit;  // heavy pairs first
    const int hk = h / G;
    const int off = p.Lkv - p.Lq;
    // Key tiles [lo[w], hi[w]) hold a key visible to some row of query tile w: all of
    // them without a mask, up to the diagonal under the causal mask, and with a
    // sliding window of W keys from the tile holding its first row's first visible
    // key (that row sees keys r' - W < c <= r', r' = r + Lkv - Lq).
    int lo[2], hi[2];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        const int qt = 2 * pi + w;
        lo[w] = hi[w] = 0;
        if (qt >= p.nQ) continue;
        if (p.causal) {
            const int maxkey = min(p.Lq, (qt + 1) * kTile) - 1 + off;
            if (maxkey < 0) continue;
            hi[w] = min(p.nK, maxkey / kTile + 1);
            if constexpr (WIN) {
                const int minkey = qt * kTile + off - p.window + 1;
                lo[w] = minkey > 0 ? minkey / kTile : 0;
            }
        } else {
            hi[w] = p.nK;
        }
    }
    // The CTA walks key tiles base, base+1, ... (index i); tile w's own iteration j
    // is index s0[w] + j.  The two ranges overlap or touch (tile B's window starts
    // at most one key tile after A's, and A's range reaches at least that far), so
    // every index below N is visited by at least one of the tiles.
    // (without a window every range starts at key tile 0: base and s0 are zero)
    const int base = WIN ? (hi[0] > lo[0] ? lo[0] : lo[1]) : 0;
    int nvis[2], s0[2];
    int N = 0;
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        nvis[w] = hi[w] - lo[w];
        s0[w] = WIN ? lo[w] - base : 0;
        if (nvis[w] > 0) N = max(N, hi[w] - base);
    }

    if (tid == 0) {
        mbar_init(&ctrl->q_full, 1);
        for (int i = 0; i < C::NK; ++i) mbar_init(&ctrl->k_full[i], 1);
        for (int i = 0; i < C::NV; ++i) mbar_init(&ctrl->v_full[i], 1);
        for (int w = 0; w < 2; ++w) {
            for (int i = 0; i < Ctrl::NR; ++i) mbar_init(&ctrl->rel[w][i], 1);
            mbar_init(&ctrl->p_full[w][0], 4);
            mbar_init(&ctrl->p_full[w][1], 4);
            ctrl->keep[w] = 0;
            ctrl->dec[w] = 0;
        }
        mbar_init(&ctrl->never, 1);
        ctrl->abort = 0;
        ctrl->v_issued = 0;
        ctrl->turn = nvis[0] > 0 ? 0 : 1;
        ctrl->active[0] = nvis[0] > 0;
        ctrl->active[1] = nvis[1] > 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(&ctrl->tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    __syncwarp();  // the set-up above diverged inside warps; bar.sync is warp-aligned
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const Watchdog wd{&ctrl->abort, p.status, p.watchdog_ns};
    if (warp >= 8) {
      regs_dec<kRegsProducer2>();
      if (warp == 8 || warp == 11) {
        // ------------------------------------------------------------ TMA producers
        // Warp 8 loads Q and the K tiles, warp 11 the V tiles (lane 0 of each), so a K
        // load never queues behind the wait for a V slot.
        const bool kq = warp == 8;
        if (lane == 0 && N > 0) {
            if (kq) {
                tma_prefetch_desc(&tq);
                tma_prefetch_desc(&tk);
            } else {
                tma_prefetch_desc(&tv);
            }
            const int zq = b * p.Hq + h, zkv = b * p.Hkv + hk;
            if (kq) {
                const int nq = (nvis[0] > 0) + (nvis[1] > 0);
                mbar_arrive_expect_tx(&ctrl->q_full, nq * C::TILE_BYTES);
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    if (nvis[w] == 0) continue;
#pragma unroll
                    for (int x = 0; x < D / 64; ++x)
                        tma_load_3d(smem + C::OFF_Q + w * C::TILE_BYTES + x * C::BOX_BYTES, &tq, &ctrl->q_full,
                                    x * 64, (2 * pi + w) * kTile, zq);
                }
            }
            // A slot is reused once every query tile that read its previous occupant is done
            // with it: K_m by QK_w(m), covered by commit m of issuer w; V_m by PV_w(m), covered
            // by commit m+1.
            constexpr int NR = Ctrl::NR;
            int issued = 0;
            auto load_k = [&](int m) -> bool {
                const int ks = m % C::NK;
                if (m >= C::NK) {
                    const int prev = m - C::NK;
#pragma unroll
                    for (int w = 0; w < 2; ++w) {
                        const int jp = prev - s0[w];  // tile w's iteration that read K_prev
                        if (jp >= 0 && jp < nvis[w] && !mbar_wait(&ctrl->rel[w][(unsigned)jp % NR], ((unsigned)jp / NR) & 1u, wd))
                            return false;
                    }
                }
                mbar_arrive_expect_tx(&ctrl->k_full[ks], C::TILE_BYTES);
#pragma unroll
                for (int x = 0; x < D / 64; ++x)
                    tma_load_3d(smem + C::OFF_K + ks * C::TILE_BYTES + x * C::BOX_BYTES, &tk, &ctrl->k_full[ks],
                                x * 64, (base + m) * kTile, zkv);
                issued = m + 1;
                return true;
            };
            auto load_v = [&](int m) -> bool {
                const int vs = m % C::NV;
                if (m >= C::NV) {
                    const int prev = m - C::NV;
#pragma unroll
                    for (int w = 0; w < 2; ++w) {
                        const int jp = prev - s0[w];  // tile w's iteration that read V_prev
                        if (jp >= 0 && jp < nvis[w] &&
                            !mbar_wait(&ctrl->rel[w][(unsigned)(jp + 1) % NR], ((unsigned)(jp + 1) / NR) & 1u, wd))
                            return false;
                    }
                    // The slot's previous copy must have landed before the slot's barrier is
                    // armed again: an issuer whose tile skipped key tile `prev` released the
                    // slot without waiting for it.
                    if (!mbar_wait(&ctrl->v_full[vs], ((unsigned)prev / C::NV) & 1u, wd)) return false;
                }
                bool need = true;
                if (p.elide_v) {
                    // V_m is needed only if a query tile keeps key tile m.  Tile w's issuer
                    // publishes its decision as dec[w] = 2(m+1) + kept; with V elision every
                    // issuer waits for v_full of V_m (loaded or not) before it passes key tile
                    // m, so dec[w] stops there.  A word that only grows, unlike a barrier phase,
                    // may be read for any key tile without having watched the earlier ones:
                    // tile B is asked only when tile A does not keep the tile.
                    need = false;
#pragma unroll
                    for (int w = 0; w < 2 && !need; ++w) {
                        const int jm = m - s0[w];
                        if (jm < 0 || jm >= nvis[w]) continue;
                        int dv = 0;
                        if (!spin_until_ge(&ctrl->dec[w], 2 * (jm + 1), dv, wd)) return false;
                        need = (dv & 1) != 0;
                    }
                }
                if (need) {
                    mbar_arrive_expect_tx(&ctrl->v_full[vs], C::TILE_BYTES);
#pragma unroll
                    for (int x = 0; x < D / 64; ++x)
                        tma_load_3d(smem + C::OFF_V + vs * C::TILE_BYTES + x * C::BOX_BYTES, &tv, &ctrl->v_full[vs],
                                    x * 64, (base + m) * kTile, zkv);
                } else {
                    mbar_arrive(&ctrl->v_full[vs]);  // completes the slot's phase without data
                }
                issued = m + 1;
                reinterpret_cast<volatile int*>(&ctrl->v_issued)[0] = m + 1;
                return true;
            };
            if (kq) {
                for (int j = 0; j < N; ++j)
                    if (!load_k(j)) break;
                mbar_wait_drain(&ctrl->q_full, 0, kDrainNs);
                for (int j = max(0, issued - C::NK); j < issued; ++j)
                    mbar_wait_drain(&ctrl->k_full[j % C::NK], (j / C::NK) & 1, kDrainNs);
            } else {
                for (int j = 0; j < N; ++j)
                    if (!load_v(j)) break;
                // every V copy before the last NV was waited for at its slot's reuse
                for (int j = max(0, issued - C::NV); j < issued; ++j)
                    mbar_wait_drain(&ctrl->v_full[j % C::NV], (j / C::NV) & 1, kDrainNs);
            }
        }
    } else if (warp == 9 || warp == 10) {
        // ------------------------------------------------------------ MMA issuers (warp 9: tile A, warp 10: tile B)
        const int w = warp - 9;
        const int n = w ? nvis[1] : nvis[0];
        if (lane == 0 && n > 0) {
            constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
            constexpr uint32_t kIdescO = idesc_bf16(128, D, false, true);
            constexpr uint32_t kTileLo = C::TILE_BYTES >> 4;
            // low descriptor words of the operand bases (offsets within a tile are added per k-step)
            const uint32_t qlo = desc_lo(smem_u32(smem + C::OFF_Q + w * C::TILE_BYTES), 16);
            const uint32_t klo = desc_lo(smem_u32(smem + C::OFF_K), 16);
            const uint32_t vlo = desc_lo(smem_u32(smem + C::OFF_V), C::BOX_BYTES);
            const uint32_t s_t = tmem + (uint32_t)w * 128u;
            const uint32_t o_t = tmem + C::O_COL + (uint32_t)w * D;
            // QK_w(j) into S_w.  With hand_over, the turn passes to the other issuer once all
            // but kQkLeft of the k-steps are queued: the other issuer then notices it, and
            // its first MMA starts, while the tensor core still works through those steps
            // (planted-70 skipping 2.076 -> 2.026 ms; LLM prefill unchanged with one step
            // left, +0.2 % with two, +1 % with three).
            constexpr int kQkLeft = 1;
            auto issue_qk = [&](int j, bool hand_over = false) {
                const uint32_t b0 = klo + (uint32_t)(j % C::NK) * kTileLo;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t o = ((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4;
                    mma_ss_split(s_t, qlo + o, b0 + o, kIdescS, kk > 0 ? 1u : 0u);
                    if (hand_over && kk == (D / 16 - 1 - kQkLeft > 0 ? D / 16 - 1 - kQkLeft : 0))
                        reinterpret_cast<volatile int*>(&ctrl->turn)[0] = 1 - w;
                }
            };
            int ncommit = 0;
            auto commit = [&]() {
                mma_commit(&ctrl->rel[w][(unsigned)ncommit % Ctrl::NR]);
                ++ncommit;
            };
            auto issue_pv_half = [&](int vs, int half, bool first) {
                const uint32_t b0 = vlo + (uint32_t)vs * kTileLo;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const int kk = half * 4 + k4;
                    mma_ts_split(o_t, s_t + kk * 8, b0 + ((kk * 2048) >> 4), kIdescO, (!first || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = (p.test_stall && w == 0) ? mbar_wait(&ctrl->never, 0, wd) : true;
            const int sw = w ? s0[1] : s0[0];  // iteration j of this tile reads K/V index sw + j
            ok = ok && mbar_wait(&ctrl->q_full, 0, wd);
            ok = ok && mbar_wait(&ctrl->k_full[sw % C::NK], (sw / C::NK) & 1, wd);
            if (ok) {
                tc_fence_after();
                issue_qk(sw);
                commit();
            }
            volatile int* turn = &ctrl->turn;
            volatile int* active = ctrl->active;
            // The two issuers alternate groups (PV_w(j) + QK_w(j+1)) so that the tensor
            // queue runs PV_A, QK_A, PV_B, QK_B, ... and the two softmaxes stay half a
            // period apart; an issuer waits for its turn only while the other is active.
            // (MMAs that two threads issue at once are interleaved by the tensor core, which
            // delays both groups: measured 24 % slower without turns.)  The wait is a tight
            // poll of the turn word -- the hand-over gaps the tensor core while it runs --
            // with the limit checked every 256 polls.
            auto take_turn = [&]() -> bool {
                if (*turn == w || !active[1 - w]) return true;
                const uint64_t t0 = globaltimer_ns();
                uint32_t it = 0;
                while (*turn != w && active[1 - w]) {
                    if ((++it & 255u) == 0) {
                        if (*wd.abort_flag) return false;
                        if (globaltimer_ns() - t0 > wd.limit_ns) {
                            *wd.abort_flag = 1;
                            atomicOr(wd.status, kStatusTimeout);
                            return false;
                        }
                    }
                }
                return true;
            };
            int npv = 0;
            unsigned long long nskip = 0;
            const long long mapbase = ((long long)(b * p.Hq + h) * p.nQ + (2 * pi + w)) * p.nK + (w ? lo[1] : lo[0]);
            for (int j = 0; j < n && ok; ++j) {
                const int ij = sw + j;
                const int vs = ij % C::NV;
                // While the softmax works on S_j: K_(j+1) for the next QK, and V_j issued.  A
                // skipped tile needs no more of V_j than that: the V producer has then consumed
                // the release of V_(j-NV), so this issuer stays within two commits of the
                // release the producer waits for next (the release ring holds NR > 2 entries).
                if (j + 1 < n && !(ok = mbar_wait(&ctrl->k_full[(ij + 1) % C::NK], ((ij + 1) / C::NK) & 1, wd))) break;
                if (!p.elide_v) {
                    int vi = 0;
                    if (!(ok = spin_until_ge(&ctrl->v_issued, ij + 1, vi, wd))) break;
                }
                // V_j is read only by a computed tile's P.V.  Whether it has landed is tested
                // now, without blocking, so that the path from P's first half to the P.V MMAs
                // holds a single barrier wait when it has (an mbarrier operation costs the
                // issuer a few hundred cycles while a softmax warp shares its scheduler).
                const bool v_landed = mbar_test_wait(&ctrl->v_full[vs], (ij / C::NV) & 1);
                // p_full[w][0], one phase per key tile: the four warps of tile w have voted and,
                // on a computed tile, stored P's first half.  The tile is kept iff one of them
                // raised keep[w] to j+1.
                if (!(ok = mbar_wait_spin(&ctrl->p_full[w][0], j & 1, wd))) break;
                const bool skip = reinterpret_cast<volatile int*>(ctrl->keep)[w] <= j;
                if (p.elide_v) reinterpret_cast<volatile int*>(ctrl->dec)[w] = 2 * (j + 1) + (skip ? 0 : 1);
                // With V elision the producer reads the decision words, which must not run
                // past a key tile whose V phase is still open, so there every tile waits for
                // V_j's phase.
                if ((!skip || p.elide_v) && !v_landed && !(ok = mbar_wait(&ctrl->v_full[vs], (ij / C::NV) & 1, wd)))
                    break;
                if (!(ok = take_turn())) break;
                tc_fence_after();
                if (!skip) issue_pv_half(vs, 0, npv == 0);
                // the tile's record, written while the tensor core works through the queued MMAs
                nskip += skip ? 1 : 0;
                if (p.skip_map) p.skip_map[mapbase + j] = skip ? 1 : 0;
                if (p.margins) {
                    const volatile float* mr = ctrl->mred[w][j & 1];
                    p.margins[mapbase + j] = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3])) * p.scale;
                }
                if (!skip) {
                    if (!(ok = mbar_wait_spin(&ctrl->p_full[w][1], npv & 1, wd))) break;
                    tc_fence_after();
                    issue_pv_half(vs, 1, npv == 0);
                    ++npv;
                }
                // the turn passes inside the group's QK, or here when the tile has no next QK
                if (j + 1 < n) issue_qk(ij + 1, true);
                else *turn = 1 - w;
                commit();       // commit j+1: PV_w(j) and QK_w(j+1)
            }
            active[w] = 0;
            *turn = 1 - w;
            if (p.skipped && nskip) atomicAdd(p.skipped, nskip);
            // the last commit covers every MMA this thread issued
            if (ncommit > 0)
                mbar_wait_drain(&ctrl->rel[w][(unsigned)(ncommit - 1) % Ctrl::NR], ((unsigned)(ncommit - 1) / Ctrl::NR) & 1u, kDrainNs);
        }
      }
    } else {
        // ------------------------------------------------------------ softmax (WG 0: tile A, WG 1: tile B)
        regs_inc<kRegsSoftmax2>();
        const int w = warp >> 2;
        const int t = tid & 127;
        const int qt = 2 * pi + w;
        const int n = w ? nvis[1] : nvis[0];
        const int lo_w = w ? lo[1] : lo[0];
        const int rabs = qt * kTile + t;
        const bool valid = rabs < p.Lq;
        const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_col = (uint32_t)w * 128u;
        const uint32_t o_col = C::O_COL + (uint32_t)w * D;
        const int lim_row = p.causal ? rabs + off : 0x3fffffff;
        float m_exact = -CUDART_INF_F, m_ref = -CUDART_INF_F, l = 0.f;
        int npv = 0;

        for (int j = 0; j < n; ++j) {
            // commit j: S_j is in TMEM and O holds PV_w(j-1)
            mbar_wait(&ctrl->rel[w][(unsigned)j % Ctrl::NR], ((unsigned)j / Ctrl::NR) & 1u, wd);
            tc_fence_after();
            // S_j with the maximum of each 32-column quarter of the row (load and reduce)
            uint32_t xr[128];
            float lm[4];
            tmem_ld32_max(tl + s_col + 0, xr, lm[0]);
            tmem_ld32_max(tl + s_col + 32, xr + 32, lm[1]);
            tmem_ld32_max(tl + s_col + 64, xr + 64, lm[2]);
            tmem_ld32_max(tl + s_col + 96, xr + 96, lm[3]);
            tmem_ld_wait();
            fence_regs<128>(xr);
            asm volatile("" : "+f"(lm[0]), "+f"(lm[1]), "+f"(lm[2]), "+f"(lm[3]));  // used after the wait
            const int kt = (lo_w + j) * kTile;  // first key of this key tile
            const int lim = min(p.Lkv - 1, lim_row) - kt;
            // sliding window: keys before r' - W + 1 are outside it
            const int lim_lo = WIN ? rabs + off - p.window + 1 - kt : 0;
            // the row's tile max: from the loads, unless a mask cuts the tile (diagonal,
            // ragged or window tiles), whose visible scores need their own maximum
            float mt;
            if (lim < kTile - 1 || lim_lo > 0) {
#pragma unroll
                for (int c = 0; c < kTile; ++c)
                    if (c > lim || c < lim_lo) xr[c] = __float_as_uint(-CUDART_INF_F);
                mt = row_max128(xr);
            } else {
                mt = fmaxf(fmaxf(lm[0], lm[1]), fmaxf(lm[2], lm[3]));
            }
            const float mnew = fmaxf(m_exact, mt);
            const float diff = mt - mnew;
            const bool vote_skip = !valid || (diff < p.thr_raw);
            if (p.margins) {
                float g = valid ? ((mt == -CUDART_INF_F && mnew == -CUDART_INF_F) ? CUDART_INF_F : diff)
                                : -CUDART_INF_F;
#pragma unroll
                for (int sh = 16; sh > 0; sh >>= 1) g = fmaxf(g, __shfl_xor_sync(0xffffffffu, g, sh));
                if (lane == 0) ctrl->mred[w][j & 1][warp & 3] = g;
            }
            // Tile vote.  A warp with a row that keeps the tile raises keep[w] to j+1 and
            // arrives at the tile's barrier without waiting; only warps whose 32 rows all
            // vote to skip wait there for the other warps.  keep[w] only grows, and key
            // tile j+1 starts after every warp has finished tile j, so it needs no reset.
            // The MMA issuer reads the same word and writes the tile's record.
            // The MMA issuer learns the decision from p_full[w][0], one phase per key tile:
            // every warp arrives on it after P's first half on a computed tile; on a skipped
            // one the first warp arrives for all four right after the decision.
            const unsigned all = __all_sync(0xffffffffu, vote_skip);
            bool skip = false;
            if (!all) {
                // every writer stores the same value j+1, so a plain store does
                st_shared_if(&ctrl->keep[w], (uint32_t)(j + 1), lane == 0);
                __syncwarp();
                named_bar_arrive(1 + w, 128);
            } else {
                tc_fence_before();  // S_j's loads are done: a skipped tile's S may be overwritten next
                named_bar_sync(1 + w, 128);
                skip = reinterpret_cast<volatile int*>(ctrl->keep)[w] <= j;
            }
            m_exact = mnew;
            if (!skip) {
                const bool move = mnew != -CUDART_INF_F && (m_ref == -CUDART_INF_F || mnew > m_ref + p.lazy_raw);
                const float alpha = move ? (m_ref == -CUDART_INF_F ? 0.f : ex2((m_ref - mnew) * p.c_log2)) : 1.f;
                if (__any_sync(0xffffffffu, move) && npv > 0) {
#pragma unroll
                    for (int cc = 0; cc < D; cc += 32) {
                        uint32_t tt[32];
                        tmem_ld32(tl + o_col + cc, tt);
                        tmem_ld_wait();
                        fence_regs<32>(tt);
#pragma unroll
                        for (int i = 0; i < 32; ++i) tt[i] = __float_as_uint(__uint_as_float(tt[i]) * alpha);
                        tmem_st32(tl + o_col + cc, tt);
                    }
                    tmem_st_wait();
                }
                if (move) {
                    l *= alpha;
                    m_ref = mnew;
                }
                const float mc = (m_ref == -CUDART_INF_F ? 0.f : m_ref) * p.c_log2;
                float rs = 0.f;
                // P in two 32-column stores (one per half; measured 1.6 % faster than four
                // 16-column ones)
#pragma unroll
                for (int ch = 0; ch < 4; ch += 2) {
                    uint32_t pk[32];
                    rs += exp_pack32(xr + ch * 32, p.c_log2, mc, pk);
                    rs += exp_pack32(xr + ch * 32 + 32, p.c_log2, mc, pk + 16);
                    tmem_st32(tl + s_col + ch * 16, pk);
                    if (ch == 0) {  // first half of P (keys 0..63) is in TMEM: let PV start on it
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        mbar_arrive_if(&ctrl->p_full[w][0], lane == 0);
                        fence_regs<64>(xr + 64);  // keep the second half's math after the signal
                    }
                }
                l += rs;
                ++npv;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                mbar_arrive_if(&ctrl->p_full[w][1], lane == 0);
            } else {
                // every warp of the tile voted to skip and left the vote barrier: the first
                // warp arrives for all four (measured 0.3-1 % faster than four arrivals)
                mbar_arrive_cnt_if(&ctrl->p_full[w][0], 4, (warp & 3) == 0 && lane == 0);
            }
        }

        if (n > 0) {  // commit n covers the last PV
            mbar_wait(&ctrl->rel[w][(unsigned)n % Ctrl::NR], ((unsigned)n / Ctrl::NR) & 1u, wd);
            tc_fence_after();
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + ((long long)(b * p.Hq + h) * p.Lq + rabs) * D;
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
            uint32_t tt[32];
            if (npv > 0) {
                tmem_ld32(tl + o_col + cc, tt);
                tmem_ld_wait();
                fence_regs<32>(tt);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) tt[i] = 0u;
            }
            if (valid) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 v4;
                    v4.x = pack_bf16x2(__uint_as_float(tt[q4 * 8 + 0]) * inv, __uint_as_float(tt[q4 * 8 + 1]) * inv);
                    v4.y = pack_bf16x2(__uint_as_float(tt[q4 * 8 + 2]) * inv, __uint_as_float(tt[q4 * 8 + 3]) * inv);
                    v4.z = pack_bf16x2(__uint_as_float(tt[q4 * 8 + 4]) * inv, __uint_as_float(tt[q4 * 8 + 5]) * inv);
                    v4.w = pack_bf16x2(__uint_as_float(tt[q4 * 8 + 6]) * inv, __uint_as_float(tt[q4 * 8 + 7]) * inv);
                    *reinterpret_cast<uint4*>(orow + cc + q4 * 8) = v4;
                }
            }
        }
        if (valid && p.lse)
            p.lse[(long long)(b * p.Hq + h) * p.Lq + rabs] = l > 0.f ? m_ref * p.scale + __logf(l) : -CUDART_INF_F;
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D>
cudaError_t launch2_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                      cudaStream_t stream) {
    using C = Prefill2Cfg<D>;
    auto kern = p.window > 0 ? prefill2_kernel<D, true> : prefill2_kernel<D, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(((p.nQ + 1) / 2) * p.B * p.Hq));
    kern<<<grid, 384, C::SMEM, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

template <int D, bool PT>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                     cudaStream_t stream) {
    using C = PrefillCfg<D, PT>;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, PT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(p.nQ * p.B * p.Hq));
    prefill_kernel<D, PT><<<grid, 192, C::SMEM, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int d, PrefillVariant v, cudaStream_t stream) {
    switch (v) {
        case PrefillVariant::kWide:
            return launch_prefill_wide(tq, tk, tv, p, d, stream);
        case PrefillVariant::kTwoTiles:
            return d == 128 ? launch2_t<128>(tq, tk, tv, p, stream) : launch2_t<64>(tq, tk, tv, p, stream);
        case PrefillVariant::kOneTilePTmem:
            return d == 128 ? launch_t<128, true>(tq, tk, tv, p, stream) : launch_t<64, true>(tq, tk, tv, p, stream);
        default:
            return d == 128 ? launch_t<128, false>(tq, tk, tv, p, stream) : launch_t<64, false>(tq, tk, tv, p, stream);
    }
}

}  // namespace blasst
