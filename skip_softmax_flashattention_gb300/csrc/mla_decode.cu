// mla_decode.cu -- skip-softmax (BLASST) decode for multi-head latent attention
// (MLA) in its absorbed form, on sm_103a.
//
// Every cached token holds ONE row of DK = 576 values (a 512-value latent vector
// followed by a 64-value rotary key) that all query heads read: the score of head
// h is scale * (q_h . row) over the 576 values and the token's value vector is the
// row's first DV = 512 values.  All heads read the same rows, as the heads of a
// GQA group read their KV head, so the heads of a sequence form the rows of every
// tile and one skip decision covers all of them x 128 keys.  The pages name MLA
// decode as the case where skipping the exponentials and the P.V products pays,
// because it can be compute-bound (Skip-Softmax design doc, "Kernel").
//
// One CTA runs one (sequence b, split s) pass over the split's key tiles in
// ascending order.  Both products run with the key dimension on the 128 TMEM
// lanes, as in the GQA decode kernel:
//   S^T_j = K_j Q^T      M = 128 keys, N = 16, 32 or 64 (heads, zero-padded), K = 576 (36 MMAs)
//   O^T_j = V_j^T P_j^T  four M = 128 blocks of the 512 value columns, N as above, K = 128 keys
// A 576-wide key tile is 144 KB, more than a ring of whole tiles leaves room for,
// so tiles stream through a ring of 64-column boxes (16 KB) and the S MMAs of a
// tile are issued box by box as the boxes land.  A kept tile's value columns are
// read a second time after its decision, in 128-column pairs of boxes: the key
// stream never waits for a decision, the second read finds the rows in L2 (they
// were read a few microseconds earlier), and a skipped tile's values are never
// read again.  (Keeping a tile's value columns in shared memory until its decision
// instead leaves room to prefetch only one more pair, and every tile then waits a
// full memory latency: measured 13 % slower on GB300.)  O stays in TMEM as one
// accumulator over the computed tiles; when a head's reference max moves, the
// softmax threads wait for the newest P.V and rescale that head's columns in place
// before the next P.V.  The per-head maxima, the same in every thread, live in
// shared memory; each thread keeps its partial row sums.
//
// Warp roles (256 threads; 384 at 64 heads per CTA, whose softmax also runs on warps
// 8-11, see MlaCfg): warps 0-3 softmax, warp 4 key loader, warp 5 issuer of
// the S MMAs and TMEM owner, warp 6 value loader, warp 7 issuer of the P.V MMAs.
// The two MMA streams have their own issuing threads, so a P.V pass waiting for a
// decision or a value pair never holds up the S MMAs that drain the key ring.
//
// Up to 16 heads the MMA N is 16, up to 32 it is 32, up to 64 it is 64.  128 heads: a
// cluster of CG = 2 CTAs runs each (sequence, split), CTA r holding heads
// [64r, 64r + 64).  The CTAs of a cluster read the same rows, so each key box is
// loaded from memory once and multicast to all of them (the entries of ring slot k are
// issued by CTA k mod CG); a slot is refilled once every CTA's MMAs have released it
// (each MMA commit arrives on the slot's barrier in every CTA), and only onto barriers
// every CTA has armed (each CTA's S issuer arms its key slots one ring ahead).  So
// every copy into a CTA is one it waits for before it exits, also when a wait gives
// up.  The value pairs, second reads that find the rows in L2, are loaded by each CTA
// for itself: sharing them tied every value slot to the slower CTA (measured 4.3 us
// per tile for the value pairs alone at 128 heads).  The tile's decision covers all
// the heads: every CTA sends its vote and margin to every other through distributed
// shared memory, and each takes the AND of the CG votes.
//
// The same kernel serves GQA/MQA decode with 32-128 query heads per KV head
// (WideShape): K and V are separate tensors of d <= 128 values per row, run at width
// 128 (a 64-wide tensor's second column box lies outside it and reads as zeros), one
// CTA (or cluster) per (sequence, KV head, split).
//
// Paged form: the cache is a pool of pages of page_size rows and a page table maps
// each page-sized run of a sequence's keys to a page (The Hitchhiker's Guide, Phase
// 08, Section 3, "Paged Attention").  A 128-key box is then fetched as 128 /
// page_size boxes (page_size < 128) or as one box inside a page; boxes past the
// end of the sequence, or with an out-of-range page index, read as zeros.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace blasst {
namespace {

constexpr unsigned long long kDrainNs = 1000000000ull;

// Row shapes: MLA reads 576-wide latent rows whose first 512 values are the values;
// wide-group GQA/MQA reads separate K and V rows of d <= 128 values (run at width 128,
// the columns past d reading as zeros).
struct MlaShape {
    static constexpr int DK = kMlaDk, DV = kMlaDv;
    static constexpr bool SEPV = false;  // values are the rows' leading DV columns
};
struct WideShape {
    static constexpr int DK = 128, DV = 128;
    static constexpr bool SEPV = true;   // values come from their own tensor
};
constexpr int BOX_BYTES = kTile * 128;   // 128 keys x 64 columns
constexpr int PAIR_BYTES = 2 * BOX_BYTES;
constexpr int NS = 4;                    // TMEM S slots
constexpr int ND = 8;                    // decision ring
constexpr uint32_t TMEM_COLS = 512;
static_assert(NS + 2 <= ND, "ring sizes");

// Layout for NPAD heads per CTA (the MMA N: 16, 32, or 64) in clusters of CG CTAs.
// Shared memory: NKB key boxes, NVP value pairs, Q, NP P buffers.  TMEM: NS S slots of
// NPAD columns, then O (VBLK blocks of NPAD columns), one accumulator over the
// computed tiles, rescaled in place when a head's reference max moves.  (Landing each
// P.V in a fresh slot and folding it into registers instead measured 4 % slower at 16
// heads and 30 % at 32.)  More value slots at the cost of key slots measured faster,
// up to the split used for NPAD = 16.  From 32 heads one P buffer frees room for key
// boxes: five at 32 heads (Q 36 KB), four at 64 (Q 72 KB).  The key stream paces these
// shapes, and the softmax of the next tile reaches its P store after the last P.V is
// done.
template <class SH, int NPAD_, int CG>
struct MlaCfg {
    static constexpr int NPAD = NPAD_;
    static constexpr int KBOX = SH::DK / 64;         // 64-column boxes per key tile
    static constexpr int VBLK = SH::DV / 128;        // 128-column value blocks (box pairs) per key tile
    static_assert(SH::DK % 64 == 0 && SH::DV % 128 == 0 && SH::DV <= SH::DK, "row layout");
    // key box / value pair rings: MLA tiles are 9 boxes + 4 pairs, wide-group tiles 2 + 1
    static constexpr int NKB = (!SH::SEPV && NPAD == 32) ? 5 : 4;
    static constexpr int NVP = SH::SEPV ? 3 : NPAD == 16 ? 4 : NPAD == 32 ? 3 : 2;
    static constexpr int NP = (!SH::SEPV && NPAD >= 32) ? 1 : 2;  // P staging buffers
    static constexpr int Q_BYTES = KBOX * NPAD * 128;
    // P^T is the B operand of the P.V MMAs.  64 heads: MN-major, [128 keys][64 heads], so
    // each thread stores its key's row in 16-byte pieces; fewer: K-major, [key half][NPAD
    // heads][64 keys].
    static constexpr bool MNP = NPAD == 64;
    // Softmax warpgroups.  64 heads per CTA split their heads over two warpgroups, warps
    // 0-3 (heads 0-31) and 8-11 (heads 32-63), which read the same TMEM lanes: each
    // thread's share of a tile's softmax (per-head maxima, exponentials, P stores, O
    // rescale) halves.  Fewer heads: one warpgroup (warps 0-3).
    static constexpr int NGRP = NPAD == 64 ? 2 : 1;
    static constexpr int HPG = NPAD / NGRP;          // heads per softmax warpgroup
    static constexpr int THREADS = NGRP == 2 ? 384 : 256;
    static constexpr int NSW = 4 * NGRP;             // softmax warps
    static constexpr int P_BYTES = 2 * NPAD * 128;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + NKB * BOX_BYTES;
    static constexpr int OFF_Q = OFF_V + NVP * PAIR_BYTES;
    static constexpr int OFF_P = OFF_Q + Q_BYTES;
    static constexpr int OFF_CTRL = OFF_P + NP * P_BYTES;
    static constexpr uint32_t O_COL = NS * NPAD;     // O block i: columns O_COL + [i*NPAD, (i+1)*NPAD)
    static_assert(O_COL + VBLK * NPAD <= TMEM_COLS, "TMEM budget");
    struct Ctrl {
        uint64_t k_full[NKB], k_empty[NKB], v_full[NVP], v_empty[NVP];
        uint64_t s_full[NS], s_free[NS], dec_full[ND], dec_free[ND];
        uint64_t p_full[NP], p_free[NP];
        uint64_t q_full, drain[2];
        uint64_t o_done[8];         // computed tile c's P.V is done (ring of 8, phase c / 8)
        uint32_t tmem_base;
        int dec[ND];
        int abort;
        alignas(16) float red[2][4][NPAD];  // per-warp tile maxima, by tile parity
        float mex[2][NPAD];         // exact running max per head, by tile parity
        float mrf[2][NPAD];         // reference max per head, by tile parity
        float alpha[NPAD];          // this tile's rescale factor per head
        alignas(16) float nmc[NPAD];  // -(reference max) * c_log2 per head for this tile's P
        float gmar[NPAD];           // this tile's margin per head
        float lred[4][NPAD];
        float inv_l[NPAD];          // 1 / l per head for the outputs
        // clusters: per decision slot, the vote of every CTA (low word: 1 = all its
        // heads skip; high word: its margin) and the barrier their arrivals complete
        uint64_t votes[ND][8];
        uint64_t vote_full[ND];
        int cl_skip;            // the cluster's decision on the current tile
    };
    static constexpr int SMEM = OFF_CTRL + (int)sizeof(Ctrl) + 1024;
    static_assert(SMEM <= 232448, "shared memory per CTA");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <class SH, int G, bool PAGED, int CG>
__global__ void __launch_bounds__(MlaCfg<SH, mla_heads_per_cta(G), CG>::THREADS, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tkv, const __grid_constant__ CUtensorMap tv,
                      const __grid_constant__ CUtensorMap tq, const DecodeParams p) {
    using C = MlaCfg<SH, mla_heads_per_cta(G), CG>;
    constexpr int DV = SH::DV, KBOX = C::KBOX, VBLK = C::VBLK;
    constexpr int NPAD = C::NPAD, NKB = C::NKB, NVP = C::NVP, NP = C::NP, P_BYTES = C::P_BYTES;
    static_assert(!(PAGED && SH::SEPV), "the paged form is built for latent rows only");
    constexpr int OFF_K = C::OFF_K, OFF_V = C::OFF_V, OFF_Q = C::OFF_Q, OFF_P = C::OFF_P;
    constexpr uint32_t O_COL = C::O_COL;
    static_assert(CG == 1 || G == NPAD, "a cluster's CTAs hold NPAD heads each");
    static_assert(!C::MNP || G == NPAD, "the MN-major P rows are written for every one of the NPAD heads");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    auto* ctrl = reinterpret_cast<typename C::Ctrl*>(smem + C::OFF_CTRL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x / CG, hk = blockIdx.y, b = blockIdx.z;
    const int zkv = b * p.Hkv + hk;      // K/V rows of this sequence's KV head
    const uint32_t rank = CG > 1 ? cluster_ctarank() : 0u;
    // this CTA's first query head: the KV head's group of p.G heads, CTA r of a cluster
    // holding [r*NPAD, (r+1)*NPAD) of it
    const int qh0 = hk * p.G + (int)rank * NPAD;
    const int dout = SH::SEPV ? p.d : DV;  // values per output row
    constexpr uint16_t kAll = (uint16_t)((1u << CG) - 1u);
    // This sequence's keys and this split's share of its tiles: [s*nT/S, (s+1)*nT/S).
    int Lb = p.Lkv;
    if (p.seq_lens) {
        const int v = p.seq_lens[b];
        Lb = min(max(v, 0), p.Lkv);
        if (tid == 0 && s == 0 && v != Lb) atomicOr(p.status, kStatusPageTable);
    }
    const int nTb = (Lb + kTile - 1) / kTile;
    const int t0 = (int)(((long long)s * nTb) / p.S);
    const int t1 = (int)(((long long)(s + 1) * nTb) / p.S);
    const int n = t1 - t0;

    if (tid == 0) {
        // a slot's release comes from the MMAs of every CTA of the cluster
        for (int i = 0; i < NKB; ++i) { mbar_init(&ctrl->k_full[i], 1); mbar_init(&ctrl->k_empty[i], CG); }
        for (int i = 0; i < NVP; ++i) { mbar_init(&ctrl->v_full[i], 1); mbar_init(&ctrl->v_empty[i], 1); }
        for (int i = 0; i < ND; ++i) mbar_init(&ctrl->vote_full[i], 1);  // own arrival + CG votes' bytes
        // the first NKB key entries are armed before any CTA of the cluster can copy
        for (int i = 0; i < min(NKB, n * KBOX); ++i) mbar_arrive_expect_tx(&ctrl->k_full[i], BOX_BYTES);
        for (int i = 0; i < NS; ++i) { mbar_init(&ctrl->s_full[i], 1); mbar_init(&ctrl->s_free[i], C::NSW); }
        for (int i = 0; i < ND; ++i) {
            mbar_init(&ctrl->dec_full[i], 1);
            mbar_init(&ctrl->dec_free[i], 2);  // released by the P.V issuer and the value loader
        }
        for (int i = 0; i < NP; ++i) { mbar_init(&ctrl->p_full[i], C::NSW); mbar_init(&ctrl->p_free[i], 1); }
        for (int i = 0; i < 8; ++i) mbar_init(&ctrl->o_done[i], 1);
        for (int g = 0; g < NPAD; ++g)
            for (int q = 0; q < 2; ++q) ctrl->mex[q][g] = ctrl->mrf[q][g] = -CUDART_INF_F;
        mbar_init(&ctrl->q_full, 1);
        mbar_init(&ctrl->drain[0], 1);
        mbar_init(&ctrl->drain[1], 1);
        ctrl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(&ctrl->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    __syncwarp();  // the set-up above diverged inside warps; bar.sync is warp-aligned
    tc_fence_before();
    if constexpr (CG > 1)
        cluster_sync_all();  // every CTA's barriers exist before any remote arrival or copy
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const Watchdog wd{&ctrl->abort, p.status, p.watchdog_ns};
    // does this CTA issue the copies of ring slot k (with CG = 1: always)
    auto issues = [&](int k) -> bool { return CG == 1 || (k % CG) == (int)rank; };
    // a loaded box: this CTA alone, or multicast to the cluster
    auto load_box = [&](uint8_t* dst, uint64_t* bar, int x, int y, const CUtensorMap* map) {
        if constexpr (CG == 1)
            tma_load_3d(dst, map, bar, x, y, zkv);
        else
            tma_load_3d_mc(dst, map, bar, x, y, zkv, kAll);
    };
    // a slot's release: a commit arriving in this CTA, or in every CTA of the cluster
    auto release = [&](uint64_t* bar) {
        if constexpr (CG == 1)
            mma_commit(bar);
        else
            mma_commit_mc(bar, kAll);
    };

    // Paged form: sub-box i of a 64-column box covers keys [i*rows, (i+1)*rows) of
    // the tile, one page run; lane i of a loader warp reads its page index once
    // per tile and issues that sub-box of every column box.
    const int nbox = PAGED ? kTile / p.rows_per_box : 1;
    // A page index is loaded well before its copy and checked only when the copy is
    // issued: a check right after the load would hold the loader warp for the whole
    // load (measured: 12 % of the paged kernel's time at 128-row pages).
    auto page_load = [&](int tile, int i) -> int {
        const int key = tile * kTile + i * p.rows_per_box;
        return (i < nbox && key < Lb) ? p.page_table[(long long)b * p.max_pages + key / p.page_size] : -1;
    };
    auto page_check = [&](int v, int tile, int i) -> int {
        const int key = tile * kTile + i * p.rows_per_box;
        if (!(i < nbox && key < Lb)) return p.num_pages;  // past the sequence: the sub-box reads as zeros
        if (v >= 0 && v < p.num_pages) return v;
        atomicOr(p.status, kStatusPageTable);
        return p.num_pages;  // out of range: zeros
    };
    // The pool is rows: page pg's row `off` is row pg * page_size + off (an out-of-range
    // page lands past the last row and reads as zeros).  Pool row of sub-box i of a tile:
    auto sub_row = [&](int pg, int tile, int i) -> int {
        return pg * p.page_size + (tile * kTile + i * p.rows_per_box) % p.page_size;
    };
    // sub-box i (rows [i*rows, (i+1)*rows) of a 64-column box) from pool row y
    auto copy_sub = [&](uint8_t* dst, uint64_t* bar, int x, int i, int y, bool mc) {
        if (CG == 1 || !mc)
            tma_load_3d(dst + i * p.rows_per_box * 128, &tkv, bar, x, y, 0);
        else
            tma_load_3d_mc(dst + i * p.rows_per_box * 128, &tkv, bar, x, y, 0, kAll);
    };
    // With up to kLane0Subs sub-boxes a box (pages of 32 rows or more) lane 0 issues
    // them all right after the slot wait, from rows gathered once a tile; smaller pages
    // issue lane by lane after the wait's broadcast.  (Issuing every copy after the
    // broadcast put a warp reconvergence between each freed slot and its copy: the
    // paged form ran 11 % slower than the contiguous one with the same addresses.)
    constexpr int kLane0Subs = 4;
    const bool lane0_issues = nbox <= kLane0Subs;

    if (warp == 4) {
        // ------------------------------------------------------------ key loader
        // Box c of tile j is ring entry e = j*KBOX + c, in slot e % NKB.  Its copy goes
        // out once every CTA released the slot's previous entry; the entry's barrier was
        // armed by the S issuer (by the set-up for the first NKB).
        if (lane == 0) {
            // this CTA's query heads, KBOX boxes of 64 columns x NPAD heads (heads past
            // Hq and columns past the row width read as zeros)
            mbar_arrive_expect_tx(&ctrl->q_full, C::Q_BYTES);
            for (int c = 0; c < KBOX; ++c)
                tma_load_3d(smem + OFF_Q + c * (NPAD * 128), &tq, &ctrl->q_full, c * 64, qh0, b);
            tma_prefetch_desc(&tkv);
            if constexpr (SH::SEPV) tma_prefetch_desc(&tv);
        }
        int last = 0;  // entries passed
        bool ok = true;
        // paged: each lane's page index is read two tiles ahead, so the load's latency
        // never sits between a freed slot and its copy
        int pg_next = (PAGED && n > 0) ? page_load(t0, lane) : 0;
        int pg_next2 = (PAGED && n > 1) ? page_load(t0 + 1, lane) : 0;
        for (int j = 0; j < n && ok; ++j) {
            int y = 0, ys[kLane0Subs];
            if constexpr (PAGED) {
                y = sub_row(page_check(pg_next, t0 + j, lane), t0 + j, lane);
#pragma unroll
                for (int i = 0; i < kLane0Subs; ++i) ys[i] = __shfl_sync(0xffffffffu, y, i);
                pg_next = pg_next2;
                pg_next2 = j + 2 < n ? page_load(t0 + j + 2, lane) : 0;
            }
            for (int c = 0; c < KBOX; ++c) {
                const int e = j * KBOX + c, ks = e % NKB;
                if (issues(ks)) {
                    uint8_t* dst = smem + OFF_K + ks * BOX_BYTES;
                    int go = 1;
                    if (lane == 0) {
                        if (e >= NKB && !mbar_wait_cluster(&ctrl->k_empty[ks], ((e / NKB) - 1) & 1, wd)) {
                            go = 0;
                        } else if constexpr (!PAGED) {
                            load_box(dst, &ctrl->k_full[ks], c * 64, (t0 + j) * kTile, &tkv);
                        } else if (lane0_issues) {
#pragma unroll
                            for (int i = 0; i < kLane0Subs; ++i)
                                if (i < nbox) copy_sub(dst, &ctrl->k_full[ks], c * 64, i, ys[i], true);
                        }
                    }
                    if (!(ok = __shfl_sync(0xffffffffu, go, 0) != 0)) break;
                    if constexpr (PAGED) {
                        if (!lane0_issues && lane < nbox) copy_sub(dst, &ctrl->k_full[ks], c * 64, lane, y, true);
                    }
                }
                last = e + 1;
            }
        }
        if constexpr (CG > 1) {  // the other CTAs' releases of the last entries arrive here
            if (lane == 0)
                for (int e = max(0, last - NKB); e < last; ++e)
                    mbar_wait_drain(&ctrl->k_empty[e % NKB], (e / NKB) & 1, kDrainNs);
        }
    } else if (warp == 6) {
        // ------------------------------------------------------------ value loader
        // pair i of the c-th computed tile is ring entry c*VBLK + i (this CTA's own copy)
        int issued = 0;
        bool ok = true;
        // paged: each lane's page index is read one tile ahead, so the load's latency
        // never sits between a decision and the tile's first value copy
        int pg_next = (PAGED && n > 0) ? page_load(t0, lane) : 0;
        for (int j = 0; j < n && ok; ++j) {
            const int pg_raw = pg_next;
            if constexpr (PAGED) pg_next = j + 1 < n ? page_load(t0 + j + 1, lane) : 0;
            int go = 0;  // 0: stop, 1: load the tile's values, 2: tile skipped
            if (lane == 0 && mbar_wait(&ctrl->dec_full[j % ND], (j / ND) & 1, wd)) {
                const bool skipped = reinterpret_cast<volatile int*>(ctrl->dec)[j % ND] != 0;
                mbar_arrive(&ctrl->dec_free[j % ND]);
                go = skipped ? 2 : 1;  // skipped: its values are not read again
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            if (go == 0) break;
            if (go == 2) continue;
            int y = 0, ys[kLane0Subs];
            if constexpr (PAGED) {
                y = sub_row(page_check(pg_raw, t0 + j, lane), t0 + j, lane);
#pragma unroll
                for (int i = 0; i < kLane0Subs; ++i) ys[i] = __shfl_sync(0xffffffffu, y, i);
            }
            for (int i = 0; i < VBLK; ++i) {
                const int e = issued, vs = e % NVP;
                int gv = 1;
                if (lane == 0) {
                    if (e >= NVP && !mbar_wait(&ctrl->v_empty[vs], ((e / NVP) - 1) & 1, wd)) {
                        gv = 0;
                    } else {
                        mbar_arrive_expect_tx(&ctrl->v_full[vs], PAIR_BYTES);
                        if constexpr (!PAGED) {
#pragma unroll
                            for (int h = 0; h < 2; ++h)
                                tma_load_3d(smem + OFF_V + vs * PAIR_BYTES + h * BOX_BYTES, SH::SEPV ? &tv : &tkv,
                                            &ctrl->v_full[vs], i * 128 + h * 64, (t0 + j) * kTile, zkv);
                        } else if (lane0_issues) {
#pragma unroll
                            for (int sb = 0; sb < kLane0Subs; ++sb)
#pragma unroll
                                for (int h = 0; h < 2; ++h)
                                    if (sb < nbox)
                                        copy_sub(smem + OFF_V + vs * PAIR_BYTES + h * BOX_BYTES, &ctrl->v_full[vs],
                                                 i * 128 + h * 64, sb, ys[sb], false);
                        }
                    }
                }
                if (!(ok = __shfl_sync(0xffffffffu, gv, 0) != 0)) break;
                if constexpr (PAGED) {
                    if (!lane0_issues && lane < nbox) {
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            copy_sub(smem + OFF_V + vs * PAIR_BYTES + h * BOX_BYTES, &ctrl->v_full[vs],
                                     i * 128 + h * 64, lane, y, false);
                    }
                }
                issued = e + 1;
            }
        }
        if (lane == 0) {
            for (int e = max(0, issued - NVP); e < issued; ++e)
                mbar_wait_drain(&ctrl->v_full[e % NVP], (e / NVP) & 1, kDrainNs);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ S issuer
        // S^T_j, box by box as the key boxes land; each box's slot is released by a
        // commit after its four MMAs.  S slot j % NS is reused once the softmax read it.
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16(128, NPAD, false, false);
            const uint32_t sK = smem_u32(smem + OFF_K), sQ = smem_u32(smem + OFF_Q);
            const int total = n * KBOX;
            int armed = min(NKB, total), consumed = 0;
            bool ok = mbar_wait(&ctrl->q_full, 0, wd);
            if (!ok) mbar_wait_drain(&ctrl->q_full, 0, kDrainNs);  // the Q copy lands before the CTA exits
            for (int j = 0; j < n && ok; ++j) {
                const int ss = j % NS;
                if (j >= NS && !(ok = mbar_wait(&ctrl->s_free[ss], ((j / NS) - 1) & 1, wd))) break;
                for (int c = 0; c < KBOX; ++c) {
                    const int e = j * KBOX + c, ks = e % NKB;
                    if (!(ok = mbar_wait(&ctrl->k_full[ks], (e / NKB) & 1, wd))) break;
                    consumed = e + 1;
                    if (e + NKB < total) {  // arm the slot's next entry before releasing this one
                        mbar_arrive_expect_tx(&ctrl->k_full[ks], BOX_BYTES);
                        armed = e + NKB + 1;
                    }
                    tc_fence_after();
                    const uint32_t kb = sK + ks * BOX_BYTES, qb = sQ + c * (NPAD * 128);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ss(tmem + ss * NPAD, desc_kmajor_sw128(kb + kk * 32), desc_kmajor_sw128(qb + kk * 32),
                               kIdescS, (c > 0 || kk > 0) ? 1u : 0u);
                    release(&ctrl->k_empty[ks]);
                }
                if (!ok) break;
                mma_commit(&ctrl->s_full[ss]);
            }
            mma_commit(&ctrl->drain[0]);
            mbar_wait_drain(&ctrl->drain[0], 0, kDrainNs);
            // copies onto entries armed but not consumed (only after a wait gave up)
            for (int e = consumed; e < armed; ++e) mbar_wait_drain(&ctrl->k_full[e % NKB], (e / NKB) & 1, kDrainNs);
        }
    } else if (warp == 7) {
        // ------------------------------------------------------------ P.V issuer
        if (lane == 0) {
            constexpr uint32_t kIdescO = idesc_bf16(128, NPAD, true, C::MNP);
            const uint32_t sV = smem_u32(smem + OFF_V), sP = smem_u32(smem + OFF_P);
            bool ok = true;
            int comp = 0;
            for (int j = 0; j < n && ok; ++j) {
                if (!(ok = mbar_wait(&ctrl->dec_full[j % ND], (j / ND) & 1, wd))) break;
                const bool skipped = reinterpret_cast<volatile int*>(ctrl->dec)[j % ND] != 0;
                mbar_arrive(&ctrl->dec_free[j % ND]);
                if (skipped) continue;
                const int pb = comp % NP;
                if (!(ok = mbar_wait(&ctrl->p_full[pb], (comp / NP) & 1, wd))) break;
                const uint32_t pbuf = sP + pb * P_BYTES;
                for (int i = 0; i < VBLK && ok; ++i) {
                    const int e = comp * VBLK + i, vs = e % NVP;
                    if (!(ok = mbar_wait(&ctrl->v_full[vs], (e / NVP) & 1, wd))) break;
                    tc_fence_after();
                    const uint32_t vb = sV + vs * PAIR_BYTES;
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk) {
                        const uint64_t adesc = desc_mnmajor_sw128(vb + kk * 2048, BOX_BYTES);
                        const uint64_t bdesc =
                            C::MNP ? desc_mnmajor_sw128(pbuf + kk * 2048, P_BYTES)
                                   : desc_kmajor_sw128(pbuf + (kk >> 2) * (NPAD * 128) + (kk & 3) * 32);
                        // O accumulates over the computed tiles
                        const uint32_t acc = (kk > 0 || comp > 0) ? 1u : 0u;
                        mma_ss(tmem + O_COL + i * NPAD, adesc, bdesc, kIdescO, acc);
                    }
                    mma_commit(&ctrl->v_empty[vs]);
                }
                if (!ok) break;
                mma_commit(&ctrl->o_done[comp % 8]);
                mma_commit(&ctrl->p_free[pb]);
                ++comp;
            }
            mma_commit(&ctrl->drain[1]);
            mbar_wait_drain(&ctrl->drain[1], 0, kDrainNs);
        }
    } else {
        // ------------------------------------------------------------ softmax (warps 0-3, and 8-11 at 64 heads)
        constexpr int NGRP = C::NGRP, NST = 128 * NGRP;  // warpgroups, threads
        // this thread's key lane (= TMEM lane) and its warpgroup's heads [hb, hb + GH)
        const int kl = tid & 127, grp = warp >> 3;
        constexpr int GH = NGRP == 2 ? C::HPG : G;
        const int hb = grp * C::HPG;
        // in each warpgroup the thread of key lane g judges and finishes head hb + g
        const bool judge = kl < GH;
        const int hj = hb + kl;
        const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        // Clear the P buffers' padding rows (heads past G); the fence before each P
        // arrival makes the zeros visible to the MMAs.
        if constexpr (!C::MNP) {
            uint4* sp = reinterpret_cast<uint4*>(smem + OFF_P);
            for (int c = kl; c < NP * P_BYTES / 16; c += 128) sp[c] = make_uint4(0, 0, 0, 0);
        }
        const long long mapbase = (long long)zkv * p.nK;
        const float cl = p.c_log2;
        // Per-head running state common to all 128 threads lives in shared memory, by
        // tile parity: mex (exact running max) and mrf (reference max) of tile j are
        // written by thread g for head g and read by everyone from tile j+1 on (after
        // that tile's first barrier).  Per thread: the scores of its key, its partial
        // row sums and its four value columns of every head.
        // O is read and written in chunks of OCH columns (heads); a warpgroup touches OH of
        // them, from its first head on
        constexpr int OCH = NPAD < 32 ? NPAD : 32;
        constexpr int OH = NGRP == 2 ? C::HPG : NPAD;
        auto o_ld = [&](uint32_t ta, uint32_t* r) {
            if constexpr (OCH == 16)
                tmem_ld16(ta, r);
            else
                tmem_ld32(ta, r);
            tmem_ld_wait();
            fence_regs<OCH>(r);
        };
        auto o_st = [&](uint32_t ta, const uint32_t* r) {
            if constexpr (OCH == 16)
                tmem_st16(ta, r);
            else
                tmem_st32(ta, r);
        };
        float lpart[GH];  // partial row sums of this warpgroup's heads
#pragma unroll
        for (int g = 0; g < GH; ++g) lpart[g] = 0.f;
        int comp = 0, cur = 1;  // mrf[cur]: the reference max as of the last tile
        unsigned long long nskip = 0;

        for (int j = 0; j < n; ++j) {
            const int ss = j % NS, q = j & 1, qp = q ^ 1;
            mbar_wait(&ctrl->s_full[ss], (j / NS) & 1, wd);
            tc_fence_after();
            const int key = (t0 + j) * kTile + kl;
            const bool key_ok = key < Lb;
            // the scores of this thread's key, one per head of its warpgroup; read again for
            // P, so the slot is released after P (nothing stays live across the decision)
            constexpr int NLD = NGRP == 2 ? C::HPG : NPAD;
            auto load_scores = [&](uint32_t* xr) {
                if constexpr (NLD == 16)
                    tmem_ld16(tl + ss * NPAD + hb, xr);
                else if constexpr (NLD == 32)
                    tmem_ld32(tl + ss * NPAD + hb, xr);
                else
                    tmem_ld64(tl + ss * NPAD + hb, xr);
                tmem_ld_wait();
                fence_regs<NLD>(xr);
            };
            {
                // Per-head max over the warp's 32 keys.  From 32 heads: one warp-wide
                // reduction (redux.sync max.f32) per head, stored by lane 0 (measured 1-2 %
                // faster than the butterfly there).  Below: a transposing butterfly, where
                // each step hands half of the remaining heads to the partner lane, so lane L
                // ends with the max of head L >> (5 - log2 G) after G - 1 + (5 - log2 G)
                // shuffles instead of 5 G.
                uint32_t xr[NLD];
                load_scores(xr);
                float v[GH];
#pragma unroll
                for (int g = 0; g < GH; ++g) v[g] = key_ok ? __uint_as_float(xr[g]) : -CUDART_INF_F;
                if constexpr (GH >= 32) {
#pragma unroll
                    for (int g = 0; g < GH; ++g) v[g] = warp_max_f32(v[g]);
                    if (lane == 0) {
#pragma unroll
                        for (int g = 0; g < GH; g += 4)
                            *reinterpret_cast<float4*>(&ctrl->red[q][warp & 3][hb + g]) =
                                make_float4(v[g], v[g + 1], v[g + 2], v[g + 3]);
                    }
                } else {
                int hl = 0;  // head index held by this lane
#pragma unroll
                for (int st = 0; st < 5; ++st) {
                    const int o = 16 >> st;
                    const int half = G >> (st + 1);  // heads handed over at this step (0: none left)
                    if (half >= 1) {
                        const bool up = (lane & o) != 0;
#pragma unroll
                        for (int k = 0; k < half; ++k) {
                            const float send = up ? v[k] : v[k + half];
                            const float keep = up ? v[k + half] : v[k];
                            v[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
                        }
                        hl += up ? half : 0;
                    } else {
                        v[0] = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], o));
                    }
                }
                constexpr int kLow = G >= 32 ? 1 : 32 / G;  // lanes holding the same head
                constexpr int kPer = G > 32 ? G / 32 : 1;    // heads held by one lane
                if ((lane & (kLow - 1)) == 0) {
#pragma unroll
                    for (int r = 0; r < kPer; ++r) ctrl->red[q][warp][hl + r] = v[r];
                }
                }
            }
            named_bar_sync(1, NST);
            // the decision: in each warpgroup the thread of key lane g judges head hb + g,
            // the barrier takes the AND
            float mn_own = -CUDART_INF_F;
            bool vote = true;
            if (judge) {
                const volatile float* rd = &ctrl->red[q][0][hj];
                const float mt = fmaxf(fmaxf(rd[0], rd[NPAD]), fmaxf(rd[2 * NPAD], rd[3 * NPAD]));
                mn_own = fmaxf(reinterpret_cast<volatile float*>(ctrl->mex[qp])[hj], mt);
                const float diff = mt - mn_own;
                vote = diff < p.thr_raw;
                ctrl->gmar[hj] = (mt == -CUDART_INF_F && mn_own == -CUDART_INF_F) ? CUDART_INF_F : diff;
                ctrl->mex[q][hj] = mn_own;
            }
            bool skip = bar_red_and(1, NST, vote);
            float margin = -CUDART_INF_F;
            if (tid == 0 && p.margins)
                for (int g = 0; g < G; ++g) margin = fmaxf(margin, reinterpret_cast<volatile float*>(ctrl->gmar)[g]);
            if constexpr (CG > 1) {
                // The decision covers the heads of every CTA of the cluster: send this
                // CTA's vote and margin to all of them, wait for theirs, take the AND and
                // the max.  Each vote is an asynchronous store that completes its bytes on
                // the receiver's barrier, which the receiver arms for CG votes (a remote
                // arrive with cluster-scope release took ~2 us here).  A CTA is never a
                // whole tile ahead of another in this exchange, so a vote slot is never
                // overwritten before it was read.
                if (tid == 0) {
                    const int slot = j % ND;
                    const uint64_t word = ((uint64_t)__float_as_uint(margin) << 32) | (skip ? 1u : 0u);
                    mbar_arrive_expect_tx(&ctrl->vote_full[slot], CG * 8);
                    for (int r = 0; r < CG; ++r)
                        st_async_cluster_u64(cluster_addr(&ctrl->votes[slot][rank], r), word,
                                             cluster_addr(&ctrl->vote_full[slot], r));
                    bool all = mbar_wait(&ctrl->vote_full[slot], (j / ND) & 1, wd);
                    float mg = -CUDART_INF_F;
                    for (int r = 0; r < CG; ++r) {
                        const uint64_t w = reinterpret_cast<volatile uint64_t*>(ctrl->votes[slot])[r];
                        all = all && (w & 1u) != 0;
                        mg = fmaxf(mg, __uint_as_float((uint32_t)(w >> 32)));
                    }
                    margin = mg;
                    reinterpret_cast<volatile int*>(&ctrl->cl_skip)[0] = all ? 1 : 0;
                }
                named_bar_sync(1, NST);
                skip = reinterpret_cast<volatile int*>(&ctrl->cl_skip)[0] != 0;
            }
            if (tid == 0) {
                // the slot is reused only after both readers of tile j - ND released it
                if (j >= ND) mbar_wait(&ctrl->dec_free[j % ND], ((j / ND) - 1) & 1, wd);
                reinterpret_cast<volatile int*>(ctrl->dec)[j % ND] = skip ? 1 : 0;
                mbar_arrive(&ctrl->dec_full[j % ND]);
                if (rank == 0) {  // one record per tile for the whole cluster
                    if (p.skip_map) p.skip_map[mapbase + t0 + j] = skip ? 1 : 0;
                    if (p.margins) p.margins[mapbase + t0 + j] = margin * p.scale;
                    nskip += skip ? 1 : 0;
                }
            }
            // the judge of head g moves its reference max (computed tiles only) and carries
            // it into this tile's buffer; the factor for O and l goes to alpha[g]
            if (judge) {
                const float mro = reinterpret_cast<volatile float*>(ctrl->mrf[qp])[hj];
                float mr = mro, a = 1.f;
                if (!skip && mn_own != -CUDART_INF_F && (mro == -CUDART_INF_F || mn_own > mro + p.lazy_raw)) {
                    a = mro == -CUDART_INF_F ? 0.f : ex2((mro - mn_own) * cl);
                    mr = mn_own;
                }
                ctrl->mrf[q][hj] = mr;
                if (!skip) {
                    ctrl->alpha[hj] = a;
                    ctrl->nmc[hj] = -((mr == -CUDART_INF_F ? 0.f : mr) * cl);
                }
            }
            if (!skip) {
                cur = q;
                const volatile float* al = ctrl->alpha;
                {
                    // the barrier that publishes alpha, mrf[q] also tells whether any head moved;
                    // then O (the P.V of the computed tiles so far) is rescaled in TMEM once
                    // the newest P.V is done
                    const bool moved = judge && reinterpret_cast<volatile float*>(ctrl->alpha)[hj] != 1.f;
                    if (bar_red_or(1, NST, moved)) {
#pragma unroll
                        for (int g = 0; g < GH; ++g) {
                            const float a = al[hb + g];
                            if (a != 1.f) lpart[g] *= a;
                        }
                        if (comp > 0) {
                            mbar_wait(&ctrl->o_done[(comp - 1) % 8], ((comp - 1) / 8) & 1, wd);
                            tc_fence_after();
#pragma unroll 1
                            for (int i = 0; i < VBLK; ++i) {
#pragma unroll
                                for (int h = 0; h < OH / OCH; ++h) {
                                    uint32_t tt[OCH];
                                    const uint32_t ta = tl + O_COL + i * NPAD + hb + h * OCH;
                                    o_ld(ta, tt);
#pragma unroll
                                    for (int c2 = 0; c2 < OCH; ++c2)
                                        tt[c2] = __float_as_uint(__uint_as_float(tt[c2]) * al[hb + h * OCH + c2]);
                                    o_st(ta, tt);
                                }
                            }
                            tmem_st_wait();
                        }
                    }
                }
                uint32_t xr[NLD];
                load_scores(xr);
                // p = 2^(s*c - m_ref*c) for every head, in place, before any store, so that
                // the loads of the per-head constants are free to run ahead
                const float* nm = ctrl->nmc + hb;  // published by the barrier above
                if constexpr (GH >= 4) {
#pragma unroll
                    for (int g = 0; g < GH; g += 4) {
                        const float4 n4 = *reinterpret_cast<const float4*>(nm + g);
                        float x[4], a[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) x[i] = key_ok ? __uint_as_float(xr[g + i]) : -CUDART_INF_F;
                        ffma2v(a[0], a[1], x[0], x[1], cl, n4.x, n4.y);
                        ffma2v(a[2], a[3], x[2], x[3], cl, n4.z, n4.w);
#pragma unroll
                        for (int i = 0; i < 4; ++i) a[i] = ex2(a[i]);
                        fadd2_acc(lpart[g], lpart[g + 1], a[0], a[1]);
                        fadd2_acc(lpart[g + 2], lpart[g + 3], a[2], a[3]);
#pragma unroll
                        for (int i = 0; i < 4; ++i) xr[g + i] = __float_as_uint(a[i]);
                    }
                } else {
#pragma unroll
                    for (int g = 0; g < GH; ++g) {
                        const float xg = key_ok ? __uint_as_float(xr[g]) : -CUDART_INF_F;
                        const float pv = ex2(fmaf(xg, cl, nm[g]));
                        lpart[g] += pv;
                        xr[g] = __float_as_uint(pv);
                    }
                }
                const int pb = comp % NP;
                if (comp >= NP) mbar_wait(&ctrl->p_free[pb], ((comp / NP) - 1) & 1, wd);
                if constexpr (C::MNP) {
                    // this key's row of 64 heads, eight 16-byte pieces, 128-byte swizzle; each
                    // warpgroup writes the pieces of its heads
                    uint8_t* prow = smem + OFF_P + pb * P_BYTES + kl * 128;
#pragma unroll
                    for (int c = 0; c < GH / 8; ++c) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(xr[8 * c + 0]), __uint_as_float(xr[8 * c + 1]));
                        w.y = pack_bf16x2(__uint_as_float(xr[8 * c + 2]), __uint_as_float(xr[8 * c + 3]));
                        w.z = pack_bf16x2(__uint_as_float(xr[8 * c + 4]), __uint_as_float(xr[8 * c + 5]));
                        w.w = pack_bf16x2(__uint_as_float(xr[8 * c + 6]), __uint_as_float(xr[8 * c + 7]));
                        const int piece = hb / 8 + c;
                        *reinterpret_cast<uint4*>(prow + ((piece ^ (kl & 7)) << 4)) = w;
                    }
                } else {
                    uint8_t* pbuf = smem + OFF_P + pb * P_BYTES + (kl >> 6) * (NPAD * 128);
                    const int cw = (kl & 63) >> 3;
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        *reinterpret_cast<unsigned short*>(pbuf + g * 128 + ((cw ^ (g & 7)) << 4) + (kl & 7) * 2) =
                            (unsigned short)(pack_bf16x2(__uint_as_float(xr[g]), 0.f) & 0xffffu);
                }
                fence_proxy_async_smem();
                tc_fence_before();  // TMEM-O: the rescaled O is stored before the next P.V
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctrl->p_full[pb]);
                ++comp;
            }
            tc_fence_before();  // the S slot's last read is done
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctrl->s_free[ss]);
        }
        named_bar_sync(1, NST);
        cur = (n - 1) & 1;  // the last tile's buffer holds every head's final reference max

        // l = sum over the 128 key lanes; O = (TMEM accumulator) / l
#pragma unroll
        for (int g = 0; g < GH; ++g) {
            float v = lpart[g];
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) v += __shfl_xor_sync(0xffffffffu, v, sh);
            if (lane == 0) ctrl->lred[warp & 3][hb + g] = v;
        }
        named_bar_sync(1, NST);
        {
            // the judge of head g finishes it (l, lse); then every thread writes its value
            // columns of its warpgroup's heads from the TMEM accumulator
            if (judge) {
                const volatile float* lr = &ctrl->lred[0][hj];
                const float l = lr[0] + lr[NPAD] + lr[2 * NPAD] + lr[3 * NPAD];
                const float mrg = reinterpret_cast<volatile float*>(ctrl->mrf[cur])[hj];
                const float lse = l > 0.f ? mrg * p.scale + __logf(l) : -CUDART_INF_F;
                ctrl->inv_l[hj] = l > 0.f ? 1.f / l : 0.f;
                const long long hq = (long long)b * p.Hq + qh0 + hj;
                if (p.S == 1) {
                    if (p.lse) p.lse[hq] = lse;
                } else {
                    p.lse_part[(long long)s * p.B * p.Hq + hq] = lse;
                }
            }
            named_bar_sync(1, NST);
            if (comp > 0) {
                mbar_wait(&ctrl->o_done[(comp - 1) % 8], ((comp - 1) / 8) & 1, wd);
                tc_fence_after();
            }
            const volatile float* il = ctrl->inv_l;
#pragma unroll 1
            for (int i = 0; i < VBLK; ++i) {
#pragma unroll
                for (int h = 0; h < OH / OCH; ++h) {
                    uint32_t tt[OCH];
                    if (comp > 0) {
                        o_ld(tl + O_COL + i * NPAD + hb + h * OCH, tt);
                    } else {
#pragma unroll
                        for (int c2 = 0; c2 < OCH; ++c2) tt[c2] = 0u;
                    }
#pragma unroll
                    for (int c2 = 0; c2 < OCH; ++c2) {
                        const int g = hb + h * OCH + c2;
                        if (g >= G) continue;
                        const float v = __uint_as_float(tt[c2]) * il[g];
                        const long long hq = (long long)b * p.Hq + qh0 + g;
                        const int col = i * 128 + kl;
                        if (col >= dout) continue;
                        if (p.S == 1)
                            reinterpret_cast<unsigned short*>(p.o)[hq * dout + col] =
                                (unsigned short)(pack_bf16x2(v, 0.f) & 0xffffu);
                        else
                            p.o_part[((long long)s * p.B * p.Hq + hq) * dout + col] = v;
                    }
                }
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
    if constexpr (CG > 1) cluster_sync_all();  // no CTA leaves while another may still reach it
}

template <class SH, int G, bool PAGED, int CG>
cudaError_t launch_gp(const CUtensorMap& tkv, const CUtensorMap& tv, const CUtensorMap& tq, const DecodeParams& p,
                      cudaStream_t stream) {
    auto kern = mla_decode_kernel<SH, G, PAGED, CG>;
    constexpr int SMEM = MlaCfg<SH, mla_heads_per_cta(G), CG>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.S * CG), (unsigned)p.Hkv, (unsigned)p.B);
    cfg.blockDim = dim3(MlaCfg<SH, mla_heads_per_cta(G), CG>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CG > 1 ? 1 : 0;
    if constexpr (CG > 1) {  // a cluster of CG CTAs of this size must fit on the GPU
        int nclusters = 0;
        e = cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (nclusters < 1) return cudaErrorInvalidConfiguration;
    }
    return cudaLaunchKernelEx(&cfg, kern, tkv, tv, tq, p);
}
template <int G, int CG>
cudaError_t launch_g(const CUtensorMap& tkv, const CUtensorMap& tq, const DecodeParams& p, cudaStream_t stream) {
    return p.page_table ? launch_gp<MlaShape, G, true, CG>(tkv, tkv, tq, p, stream)
                        : launch_gp<MlaShape, G, false, CG>(tkv, tkv, tq, p, stream);
}

}  // namespace

// Hq <= 64: one CTA per (sequence, split); 128: clusters of 2 CTAs of 64 heads.
cudaError_t launch_mla_decode(const CUtensorMap& tkv, const CUtensorMap& tq, const DecodeParams& p,
                              cudaStream_t stream) {
    switch (p.Hq) {
        case 1: return launch_g<1, 1>(tkv, tq, p, stream);
        case 2: return launch_g<2, 1>(tkv, tq, p, stream);
        case 4: return launch_g<4, 1>(tkv, tq, p, stream);
        case 8: return launch_g<8, 1>(tkv, tq, p, stream);
        case 16: return launch_g<16, 1>(tkv, tq, p, stream);
        case 32: return launch_g<32, 1>(tkv, tq, p, stream);
        case 64: return launch_g<64, 1>(tkv, tq, p, stream);
        case 128: return launch_g<64, 2>(tkv, tq, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

// GQA/MQA decode with G = 32, 64 or 128 query heads per KV head (contiguous cache).
cudaError_t launch_wide_decode(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                               const DecodeParams& p, cudaStream_t stream) {
    switch (p.G) {
        case 32: return launch_gp<WideShape, 32, false, 1>(tk, tv, tq, p, stream);
        case 64: return launch_gp<WideShape, 64, false, 1>(tk, tv, tq, p, stream);
        case 128: return launch_gp<WideShape, 64, false, 2>(tk, tv, tq, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace blasst
