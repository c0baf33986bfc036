// prefill_wide.cu -- skip-softmax (BLASST) prefill with two query tiles per CTA and
// eight softmax warps per query tile (selected with BLASST_PREFILL_WIDE).
//
// Same pipeline as the two-tile kernel in prefill.cu (one TMA producer, one MMA
// issuer per query tile taking turns and committing once per key tile, P in TMEM),
// but each query row is handled by
// two threads: warps 0-3 own key columns 0..63 of the rows of tile A, warps 4-7
// columns 64..127; warps 8-15 do the same for tile B.  Each thread therefore takes
// the max and the exponentials of 64 scores instead of 128, which halves the
// softmax latency that sits between one tile's QK and its PV.
//
// The BLASST test per row, m~ - m_new < ln(lambda) with m_new = max(m, m~)
// (Skip-Softmax design doc, "Algorithm"; BLASST talk notes, Eq. 2), is decided by
// each column half on its own: for lambda <= 1 it holds exactly when both halves'
// maxima satisfy m~_h < m + ln(lambda) (if m~ > m the left side is 0 and the test
// fails; otherwise m_new = m).  So one barrier per tile carries both the AND of the
// votes (warp __all, then a shared-memory atomicAnd per warp, as in the BLASST
// skip-predicate reduction) and the exchange of the half maxima.
//
// Warps 16-19: warp 16 TMA producer, warps 17 / 18 MMA issuers of tiles A / B,
// warp 19 idle.  Registers: 96 per thread at launch; the producer warpgroup drops
// to 56 and the softmax warpgroups rise to 104 (4*128*104 + 128*56 = 640*96).
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace blasst {
namespace {

constexpr unsigned long long kDrainNs = 1000000000ull;
constexpr int kThreads = 640;
constexpr int kRegsLaunch = 96, kRegsSoftmax = 104, kRegsProducer = 56;
static_assert(4 * 128 * kRegsSoftmax + 128 * kRegsProducer <= kThreads * kRegsLaunch, "register split");

template <int NK, int NV>
struct WideCtrl {
    // commit c of issuer w (after QK_w(c) and PV_w(c-1)) arrives on rel[w][c % NR]:
    // S ready for the softmax, K/V slots free for the producer (as in prefill.cu)
    static constexpr int NR = (NK > NV ? NK : NV) + 1;
    uint64_t q_full;
    uint64_t k_full[NK], v_full[NV];
    uint64_t rel[2][NR];
    uint64_t p_full[2][2];
    uint64_t never;
    uint32_t tmem_base;
    int vote[2][3];
    int dec[2];
    int abort;
    int turn;
    int active[2];
    // [tile][column half][row]: the half's tile max, read by the other half; after the
    // last tile each thread writes its row sum into the other half's slot (only it
    // reads that slot), so the same words carry the row-sum exchange
    float mx[2][2][128];
    float mred[2][2][8];
};

template <int D>
struct WideCfg {
    static constexpr int TILE_BYTES = kTile * D * 2;
    static constexpr int BOX_BYTES = kTile * 128;
    static constexpr int NK = (D == 128) ? 3 : 4;
    static constexpr int NV = (D == 128) ? 2 : 4;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = 2 * TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NK * TILE_BYTES;
    static constexpr int OFF_CTRL = OFF_V + NV * TILE_BYTES;
    using Ctrl = WideCtrl<NK, NV>;
    static constexpr int SMEM = OFF_CTRL + (int)sizeof(Ctrl);  // base is 1024-aligned (checked)
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t O_COL = 256;
};


// Maximum of 64 fp32 values held as raw bits (tree of 3-input maxima).
__device__ __forceinline__ float row_max64(const uint32_t* x) {
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float* f = reinterpret_cast<const float*>(x + 8 * i);
        m[i] = fmax3(fmax3(f[0], f[1], f[2]), fmax3(f[3], f[4], f[5]), fmaxf(f[6], f[7]));
    }
    return fmax3(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_wide_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const PrefillParams p) {
    using C = WideCfg<D>;
    using Ctrl = typename C::Ctrl;
    extern __shared__ __align__(1024) uint8_t smem[];
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + C::OFF_CTRL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The 128-byte-swizzled tiles need a 1024-byte aligned base; there is no room for
    // padding, so a misaligned base ends the CTA (uniformly, before any barrier).
    if (smem_u32(smem) & 1023u) {
        if (tid == 0) atomicOr(p.status, kStatusMisaligned);
        return;
    }

    const int G = p.Hq / p.Hkv;
    const int npairs = (p.nQ + 1) >> 1;
    int unit, b, h;
    prefill_cta_coords(p, npairs, unit, b, h);
    const int pi = p.causal ? (npairs - 1 - unit) : unit;  // heavy pairs first
    const int hk = h / G;
    const int off = p.Lkv - p.Lq;
    int nvis[2];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        const int qt = 2 * pi + w;
        if (qt >= p.nQ) {
            nvis[w] = 0;
        } else if (p.causal) {
            const int maxkey = min(p.Lq, (qt + 1) * kTile) - 1 + off;
            nvis[w] = maxkey < 0 ? 0 : min(p.nK, maxkey / kTile + 1);
        } else {
            nvis[w] = p.nK;
        }
    }
    const int N = max(nvis[0], nvis[1]);

    if (tid == 0) {
        mbar_init(&ctrl->q_full, 1);
        for (int i = 0; i < C::NK; ++i) mbar_init(&ctrl->k_full[i], 1);
        for (int i = 0; i < C::NV; ++i) mbar_init(&ctrl->v_full[i], 1);
        for (int w = 0; w < 2; ++w) {
            for (int i = 0; i < Ctrl::NR; ++i) mbar_init(&ctrl->rel[w][i], 1);
            mbar_init(&ctrl->p_full[w][0], 4);
            mbar_init(&ctrl->p_full[w][1], 4);
            ctrl->vote[w][0] = ctrl->vote[w][1] = ctrl->vote[w][2] = 1;
        }
        mbar_init(&ctrl->never, 1);
        ctrl->abort = 0;
        ctrl->turn = nvis[0] > 0 ? 0 : 1;
        ctrl->active[0] = nvis[0] > 0;
        ctrl->active[1] = nvis[1] > 0;
        fence_mbar_init();
    }
    if (warp == 17) {
        tmem_alloc(&ctrl->tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    __syncwarp();  // the set-up above diverged inside warps; bar.sync is warp-aligned
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const Watchdog wd{&ctrl->abort, p.status, p.watchdog_ns};

    if (warp >= 16) {
        regs_dec<kRegsProducer>();
        if (warp == 16) {
            // -------------------------------------------------------- TMA producer
            if (lane == 0 && N > 0) {
                tma_prefetch_desc(&tq);
                tma_prefetch_desc(&tk);
                tma_prefetch_desc(&tv);
                const int zq = b * p.Hq + h, zkv = b * p.Hkv + hk;
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
                // a slot is reused once every query tile that read its previous occupant is done
                // with it: K_m by QK_w(m) (commit m), V_m by PV_w(m) (commit m+1)
                constexpr int NR = Ctrl::NR;
                int issued_k = 0, issued_v = 0;
                for (int j = 0; j < N; ++j) {
                    const int ks = j % C::NK;
                    bool okk = true;
                    if (j >= C::NK) {
                        const int prev = j - C::NK;
                        for (int w = 0; w < 2 && okk; ++w)
                            if (prev < nvis[w]) okk = mbar_wait(&ctrl->rel[w][(unsigned)prev % NR], ((unsigned)prev / NR) & 1u, wd);
                    }
                    if (!okk) break;
                    mbar_arrive_expect_tx(&ctrl->k_full[ks], C::TILE_BYTES);
#pragma unroll
                    for (int x = 0; x < D / 64; ++x)
                        tma_load_3d(smem + C::OFF_K + ks * C::TILE_BYTES + x * C::BOX_BYTES, &tk, &ctrl->k_full[ks],
                                    x * 64, j * kTile, zkv);
                    issued_k = j + 1;
                    const int vs = j % C::NV;
                    bool okv = true;
                    if (j >= C::NV) {
                        const int prev = j - C::NV;
                        for (int w = 0; w < 2 && okv; ++w)
                            if (prev < nvis[w])
                                okv = mbar_wait(&ctrl->rel[w][(unsigned)(prev + 1) % NR], ((unsigned)(prev + 1) / NR) & 1u, wd);
                    }
                    if (!okv) break;
                    mbar_arrive_expect_tx(&ctrl->v_full[vs], C::TILE_BYTES);
#pragma unroll
                    for (int x = 0; x < D / 64; ++x)
                        tma_load_3d(smem + C::OFF_V + vs * C::TILE_BYTES + x * C::BOX_BYTES, &tv, &ctrl->v_full[vs],
                                    x * 64, j * kTile, zkv);
                    issued_v = j + 1;
                }
                mbar_wait_drain(&ctrl->q_full, 0, kDrainNs);
                for (int j = max(0, issued_k - C::NK); j < issued_k; ++j)
                    mbar_wait_drain(&ctrl->k_full[j % C::NK], (j / C::NK) & 1, kDrainNs);
                for (int j = max(0, issued_v - C::NV); j < issued_v; ++j)
                    mbar_wait_drain(&ctrl->v_full[j % C::NV], (j / C::NV) & 1, kDrainNs);
            }
        } else if (warp == 17 || warp == 18) {
            // -------------------------------------------------------- MMA issuers
            const int w = warp - 17;
            const int n = nvis[w];
            if (lane == 0 && n > 0) {
                constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
                constexpr uint32_t kIdescO = idesc_bf16(128, D, false, true);
                constexpr uint32_t kTileLo = C::TILE_BYTES >> 4;
                const uint32_t qlo = desc_lo(smem_u32(smem + C::OFF_Q + w * C::TILE_BYTES), 16);
                const uint32_t klo = desc_lo(smem_u32(smem + C::OFF_K), 16);
                const uint32_t vlo = desc_lo(smem_u32(smem + C::OFF_V), C::BOX_BYTES);
                const uint32_t s_t = tmem + (uint32_t)w * 128u;
                const uint32_t o_t = tmem + C::O_COL + (uint32_t)w * D;
                auto issue_qk = [&](int j) {
                    const uint32_t b0 = klo + (uint32_t)(j % C::NK) * kTileLo;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = ((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4;
                        mma_ss_split(s_t, qlo + o, b0 + o, kIdescS, kk > 0 ? 1u : 0u);
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
                        mma_ts_split(o_t, s_t + kk * 8, b0 + ((kk * 2048) >> 4), kIdescO,
                                     (!first || kk > 0) ? 1u : 0u);
                    }
                };
                volatile int* turn = &ctrl->turn;
                volatile int* active = ctrl->active;
                // Groups (PV_w(j) + QK_w(j+1)) of the two issuers alternate in the tensor
                // queue, which keeps the two tiles' softmaxes half a period apart.  The turn
                // word is polled tightly (the limit is checked every 256 polls) and handed
                // over before the commit, as in the default kernel.
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
                bool ok = (p.test_stall && w == 0) ? mbar_wait(&ctrl->never, 0, wd) : true;
                ok = ok && mbar_wait(&ctrl->q_full, 0, wd);
                ok = ok && mbar_wait(&ctrl->k_full[0], 0, wd);
                if (ok) {
                    tc_fence_after();
                    issue_qk(0);
                    commit();
                }
                int npv = 0;
                for (int j = 0; j < n && ok; ++j) {
                    const int vs = j % C::NV;
                    if (j + 1 < n &&
                        !(ok = mbar_wait(&ctrl->k_full[(j + 1) % C::NK], ((j + 1) / C::NK) & 1, wd)))
                        break;
                    const bool v_landed = mbar_test_wait(&ctrl->v_full[vs], (j / C::NV) & 1);
                    if (!(ok = mbar_wait_spin(&ctrl->p_full[w][0], j & 1, wd))) break;
                    const bool skip = reinterpret_cast<volatile int*>(ctrl->dec)[w] != 0;
                    // V_j must have landed before its slot is released, also when the tile is skipped
                    if (!v_landed && !(ok = mbar_wait(&ctrl->v_full[vs], (j / C::NV) & 1, wd))) break;
                    if (!(ok = take_turn())) break;
                    tc_fence_after();
                    if (!skip) issue_pv_half(vs, 0, npv == 0);
                    if (!(ok = mbar_wait_spin(&ctrl->p_full[w][1], j & 1, wd))) break;
                    tc_fence_after();
                    if (!skip) {
                        issue_pv_half(vs, 1, npv == 0);
                        ++npv;
                    }
                    if (j + 1 < n) issue_qk(j + 1);
                    *turn = 1 - w;
                    commit();  // commit j+1: PV_w(j) and QK_w(j+1)
                }
                active[w] = 0;
                *turn = 1 - w;
                if (ncommit > 0)  // the last commit covers every MMA of this thread
                    mbar_wait_drain(&ctrl->rel[w][(unsigned)(ncommit - 1) % Ctrl::NR],
                                    ((unsigned)(ncommit - 1) / Ctrl::NR) & 1u, kDrainNs);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax
        regs_inc<kRegsSoftmax>();
        const int w = warp >> 3;          // query tile
        const int half = (warp >> 2) & 1; // key columns 64*half .. 64*half+63
        const int r = ((warp & 3) << 5) | lane;  // row within the tile = TMEM lane
        const int tt = tid & 255;         // thread index within the tile's 256 threads
        const int qt = 2 * pi + w;
        const int n = nvis[w];
        const int rabs = qt * kTile + r;
        const bool valid = rabs < p.Lq;
        const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_col = (uint32_t)w * 128u + (uint32_t)half * 64u;  // this thread's S columns
        const uint32_t p_col = (uint32_t)w * 128u + (uint32_t)half * 32u;  // this thread's P columns
        const uint32_t o_col = C::O_COL + (uint32_t)w * D + (uint32_t)half * (D / 2);
        const int lim_row = p.causal ? rabs + off : 0x3fffffff;
        const long long mapbase = ((long long)(b * p.Hq + h) * p.nQ + qt) * p.nK;
        float m_exact = -CUDART_INF_F, m_ref = -CUDART_INF_F, l = 0.f;
        int npv = 0;
        unsigned long long nskip = 0;
        int* vote = ctrl->vote[w];

        for (int j = 0; j < n; ++j) {
            // commit j: S_j is in TMEM and O holds PV_w(j-1)
            mbar_wait(&ctrl->rel[w][(unsigned)j % Ctrl::NR], ((unsigned)j / Ctrl::NR) & 1u, wd);
            tc_fence_after();
            // this thread's 64 scores with the maximum of each 32-column half (load and reduce)
            uint32_t xr[64];
            float lm[2];
            tmem_ld32_max(tl + s_col, xr, lm[0]);
            tmem_ld32_max(tl + s_col + 32, xr + 32, lm[1]);
            tmem_ld_wait();
            fence_regs<64>(xr);
            asm volatile("" : "+f"(lm[0]), "+f"(lm[1]));  // used after the wait
            const int lim = min(p.Lkv - 1, lim_row) - j * kTile - half * 64;
            float mth;
            if (lim < 63) {  // a mask cuts the tile: the visible scores need their own maximum
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c > lim) xr[c] = __float_as_uint(-CUDART_INF_F);
                mth = row_max64(xr);
            } else {
                mth = fmaxf(lm[0], lm[1]);
            }
            ctrl->mx[w][half][r] = mth;
            // this half's vote; the row votes "skip" iff both halves do (see the header)
            const bool vote_skip = !valid || (mth < m_exact + p.thr_raw);
            const unsigned all = __all_sync(0xffffffffu, vote_skip);
            if (lane == 0) atomicAnd(&vote[j % 3], (int)all);
            named_bar_sync(1 + w, 256);
            const bool skip = reinterpret_cast<volatile int*>(vote)[j % 3] != 0;
            const float mt = fmaxf(mth, reinterpret_cast<volatile float*>(ctrl->mx[w][half ^ 1])[r]);
            const float mnew = fmaxf(m_exact, mt);
            if (p.margins) {
                const float diff = mt - mnew;
                float g = valid ? ((mt == -CUDART_INF_F && mnew == -CUDART_INF_F) ? CUDART_INF_F : diff)
                                : -CUDART_INF_F;
#pragma unroll
                for (int sh = 16; sh > 0; sh >>= 1) g = fmaxf(g, __shfl_xor_sync(0xffffffffu, g, sh));
                if (lane == 0) ctrl->mred[w][j & 1][warp & 7] = g;
                named_bar_sync(1 + w, 256);
            }
            if (tt == 0) {
                vote[(j + 2) % 3] = 1;
                reinterpret_cast<volatile int*>(ctrl->dec)[w] = skip ? 1 : 0;
                if (p.skip_map) p.skip_map[mapbase + j] = skip ? 1 : 0;
                if (p.margins) {
                    const volatile float* mr = ctrl->mred[w][j & 1];
                    float g = mr[0];
#pragma unroll
                    for (int k = 1; k < 8; ++k) g = fmaxf(g, mr[k]);
                    p.margins[mapbase + j] = g * p.scale;
                }
                nskip += skip ? 1 : 0;
            }
            m_exact = mnew;
            if (!skip) {
                // move the reference max (rarely, see lazy_raw); P uses the new one
                const bool move = mnew != -CUDART_INF_F && (m_ref == -CUDART_INF_F || mnew > m_ref + p.lazy_raw);
                const float alpha = move ? (m_ref == -CUDART_INF_F ? 0.f : ex2((m_ref - mnew) * p.c_log2)) : 1.f;
                if (move) m_ref = mnew;
                const float mc = (m_ref == -CUDART_INF_F ? 0.f : m_ref) * p.c_log2;
                float rs = 0.f;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t pk[8];
                    rs += exp_pack16(xr + ch * 16, p.c_log2, mc, pk);
                    tmem_st8(tl + p_col + ch * 8, pk);
                }
                // rescale this half-row of O to the new reference before its PV is issued
                if (__any_sync(0xffffffffu, move) && npv > 0) {
#pragma unroll
                    for (int cc = 0; cc < D / 2; cc += 16) {
                        uint32_t ov[16];
                        tmem_ld16(tl + o_col + cc, ov);
                        tmem_ld_wait();
                        fence_regs<16>(ov);
#pragma unroll
                        for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st16(tl + o_col + cc, ov);
                    }
                }
                l = l * alpha + rs;
                ++npv;
                tmem_st_wait();
                tc_fence_before();
            }
            __syncwarp();
            mbar_arrive_if(&ctrl->p_full[w][half], lane == 0);
        }

        // ---------------------------------------------------------------- epilogue
        if (n > 0) {  // commit n covers the last PV
            mbar_wait(&ctrl->rel[w][(unsigned)n % Ctrl::NR], ((unsigned)n / Ctrl::NR) & 1u, wd);
            tc_fence_after();
        }
        ctrl->mx[w][half ^ 1][r] = l;
        named_bar_sync(1 + w, 256);
        const float lt = l + reinterpret_cast<volatile float*>(ctrl->mx[w][half])[r];
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + ((long long)(b * p.Hq + h) * p.Lq + rabs) * D +
                         half * (D / 2);
#pragma unroll
        for (int cc = 0; cc < D / 2; cc += 16) {
            uint32_t ov[16];
            if (npv > 0) {
                tmem_ld16(tl + o_col + cc, ov);
                tmem_ld_wait();
                fence_regs<16>(ov);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) ov[i] = 0u;
            }
            if (valid) {
#pragma unroll
                for (int q4 = 0; q4 < 2; ++q4) {
                    uint4 v4;
                    v4.x = pack_bf16x2(__uint_as_float(ov[q4 * 8 + 0]) * inv, __uint_as_float(ov[q4 * 8 + 1]) * inv);
                    v4.y = pack_bf16x2(__uint_as_float(ov[q4 * 8 + 2]) * inv, __uint_as_float(ov[q4 * 8 + 3]) * inv);
                    v4.z = pack_bf16x2(__uint_as_float(ov[q4 * 8 + 4]) * inv, __uint_as_float(ov[q4 * 8 + 5]) * inv);
                    v4.w = pack_bf16x2(__uint_as_float(ov[q4 * 8 + 6]) * inv, __uint_as_float(ov[q4 * 8 + 7]) * inv);
                    *reinterpret_cast<uint4*>(orow + cc + q4 * 8) = v4;
                }
            }
        }
        if (valid && half == 0 && p.lse)
            p.lse[(long long)(b * p.Hq + h) * p.Lq + rabs] = lt > 0.f ? m_ref * p.scale + __logf(lt) : -CUDART_INF_F;
        if (tt == 0 && p.skipped && nskip) atomicAdd(p.skipped, nskip);
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 17) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D>
cudaError_t launch_wide_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const PrefillParams& p, cudaStream_t stream) {
    using C = WideCfg<D>;
    cudaError_t e =
        cudaFuncSetAttribute(prefill_wide_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(((p.nQ + 1) / 2) * p.B * p.Hq));
    prefill_wide_kernel<D><<<grid, kThreads, C::SMEM, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_wide(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const PrefillParams& p, int d, cudaStream_t stream) {
    return d == 128 ? launch_wide_t<128>(tq, tk, tv, p, stream) : launch_wide_t<64>(tq, tk, tv, p, stream);
}

}  // namespace blasst
