// bf16 m-grouped SwiGLU expert FFN on CTA pairs (tcgen05 cta_group::2).
//
// Same contract as grouped_tc.cu (page "Expert Parallelism (EP)",
// llm-infra-atlas, sections 1-2: the routed experts' fc1 -> act -> fc2 as
// m-grouped GEMMs over the expert-contiguous layout; weight shapes of
// "Expert Tensor Parallel design" section 4.3), built for the way the
// 5th-generation tensor cores share operands across two SMs:
//
//   * a cluster of two CTAs (one SM each) computes a 256-row x 256-column
//     tile of one expert with tcgen05.mma.cta_group::2 (M=256, N=256, K=16):
//     each CTA holds its own 128 rows of A and half of B (128 rows), so per
//     SM the operands that TMA writes and the MMA reads from shared memory
//     are 32 KB per k-step instead of 48 KB for a 128x256 single-SM tile;
//     measured with L2-resident weights, the MMA issuer waits for operands
//     15% of the time here against 27% with single-SM tiles;
//   * GEMM1: CTA r holds rows n0+64r .. n0+64r+63 of w1 followed by the same
//     rows of w3, so the pair's N=256 columns are [gate, up] of hidden units
//     n0..n0+63 and then of n0+64..n0+127; the epilogue pairs column c with
//     c+64 and writes h = SiLU(gate) * up directly.  GEMM2: the two CTAs hold
//     consecutive 128-row halves of a 256-row w2 tile and store y in fp16
//     (the fp32 accumulator rounded once; a value beyond the fp16 range
//     raises FLAG_RANGE);
//   * an expert's last tile with at most 128 valid rows runs as an M=128
//     pair MMA (64 rows per CTA) instead of M=256, so segments are padded to
//     128 rows as with single-SM tiles.  With M=128 each CTA's 64 rows sit in
//     TMEM lanes 0-63 for the first half of N and again in lanes 64-127 for
//     the second half (128 TMEM columns; determined on GB300 with a probe);
//   * the leader CTA (rank 0) issues the MMAs; both producers' TMA loads
//     complete on the leader's "full" barrier; the leader's commits arrive
//     on both CTAs' "empty" / "tmem full" barriers (multicast); both
//     epilogues release the leader's "tmem empty" barrier;
//   * six 32 KB pipeline stages, two TMEM accumulators of 256 columns;
//   * every mbarrier wait is bounded (FLAG_TIMEOUT); the pair meets at a
//     cluster barrier before TMEM is freed;
//   * both GEMMs run in ONE persistent cooperative launch: all GEMM1 tiles,
//     then all GEMM2 tiles, in one static round-robin order.  GEMM1 epilogue
//     warps count finished tiles per 256-row block in a workspace counter
//     (release); a producer waits for its block's count (acquire, bounded)
//     before its first TMA load of h, so GEMM2 starts block by block while
//     the last GEMM1 tiles still run, and the prologue (tile table, TMEM,
//     barriers) is paid once.  Every tile depends only on tiles earlier in
//     the order and the cooperative launch keeps all CTAs resident, so the
//     waits end.  The last CTA to finish zeroes the counters.  Where the
//     device refuses a cooperative cluster launch, the GEMMs run as two
//     launches.  (Interleaving GEMM2 tiles of block b between GEMM1 tiles of
//     later blocks, to overlap the tensor-bound and the HBM-bound phase, was
//     measured slower on GB300: fine-grained 0.379 vs 0.360 ms, DeepSeek-V3-
//     shaped 5.78 vs 5.45 ms.)
#include <cuda.h>

#include <algorithm>
#include <cstdlib>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int P_BM = 128;                        // rows per CTA
constexpr int P_PAIR_M = 2 * P_BM;               // rows per pair tile
constexpr int P_BN = 256;                        // N of the pair MMA
constexpr int P_BK = 64;
// GEMM2's y through shared memory and TMA stores (1) or straight from
// registers (0); the staging takes one ring stage's worth of smem.
#ifndef MOE_PAIR_TMA_Y
#define MOE_PAIR_TMA_Y 1
#endif
#ifndef MOE_PAIR_STAGES
#define MOE_PAIR_STAGES (MOE_PAIR_TMA_Y ? 5 : 6)
#endif
constexpr int P_STAGES = MOE_PAIR_STAGES;
constexpr int P_A_BYTES = P_BM * P_BK * 2;       // 16 KB
constexpr int P_B_BYTES = (P_BN / 2) * P_BK * 2; // 16 KB: this CTA's half of B
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
constexpr int P_EPI_WARPS = 4;
// Gather mode (a separate instantiation): GEMM1's A rows come straight
// from x by token_of_row, copied by extra warps instead of TMA-loaded from
// x_perm.
constexpr int P_GATHER_WARPS = 4;  // one per stage in flight (stage n: warp n % 4)
// The MMA warp's wait on a stage with gathered rows acquires at cluster
// scope (1) or CTA scope (0).
#ifndef MOE_GATHER_ACQ_CLUSTER
#define MOE_GATHER_ACQ_CLUSTER 1
#endif
constexpr int pair_threads(bool gather) {
    return 64 + 32 * P_EPI_WARPS + (gather ? 32 * P_GATHER_WARPS : 0);
}
constexpr int P_ACC_COLS = 256;
constexpr int P_TMEM_COLS = 512;
constexpr int P_NBARS = 24;
// An expert's last tile with at most P_SWAP_MAX valid rows runs transposed:
// the weights are the M=256 operand and the tile's tokens the N operand
// (N = valid rows rounded up to 32), so the MMA time follows the valid rows.
// (An M=128 pair MMA takes as long as an M=256 one on GB300.)  Measured on
// GB300: with at most 32 rows, DeepSeek-V3-shaped (tails of a few rows)
// 4.97 vs 5.01 ms; raising the limit to 128 makes the fine-grained call
// slower (0.40 vs 0.356 ms), because a transposed tile still streams a full
// 128-row weight slice per k-step and its epilogue writes one row per
// 32-lane store.
#ifndef MOE_PAIR_SWAP_MAX
#define MOE_PAIR_SWAP_MAX 32
#endif
constexpr int P_SWAP_MAX = MOE_PAIR_SWAP_MAX;
static_assert(P_SWAP_MAX <= P_PAIR_M, "a transposed tile holds at most 256 tokens");
constexpr int P_XBUF_BYTES = 2 * 32 * 32 * 4;  // GEMM1 transposed tiles: up -> gate handoff
// GEMM2 y staging: per epilogue warp two boxes of 32 rows x 64 fp16 (128-byte swizzle)
constexpr int P_YBOX_BYTES = 32 * 64 * 2;
constexpr int P_YSTAGE_BYTES = MOE_PAIR_TMA_Y ? P_EPI_WARPS * 2 * P_YBOX_BYTES : 0;


// Tile schedules.
enum : int {
    SCHED_GEMM1 = 0,  // GEMM1 tiles only: h = SiLU(x w1^T) * (x w3^T)
    SCHED_GEMM2 = 1,  // GEMM2 tiles only: y = h w2^T
    SCHED_BOTH = 2,   // all GEMM1 tiles, then all GEMM2 tiles (per-block dependency)
};

struct PairParams {
    int sched;
    int E_local, e_first;
    int rows_alloc;
    int nk0, nk1;         // k-blocks of GEMM1 (K = D) and GEMM2 (K = H_local)
    int nt0, nt1;         // output tiles along N: 128 h columns (GEMM1), 256 y columns (GEMM2)
    int n_out0, n_out1;   // H_local, D
    const int *seg_off;
    const int *tpe;
    void *out0;           // bf16 h [rows, H_local]
    __nv_bfloat16 *gu_out;  // training forward: g | u pre-activations [rows, 2 H_local] (or null)
    // FP8 GEMM1: x_perm, w1 and w3 are e4m3 codes (K blocks of 128 per stage)
    // with one scale per row of x_perm and per row of w1 / w3 ([E_local, H_local])
    int g1_fp8;
    const float *x_scale, *w1_scale, *w3_scale;
    // Combine fused into GEMM2: its epilogue adds w * y for each row into
    // comb [T, n_out1] (fp32 atomics; the token and slot weight of row r from
    // token_of_row, row_of [T, k] and topk_w) instead of storing y_perm
    float *comb;
    // Gather mode (the kGather instantiation, bf16 GEMM1): A rows of GEMM1
    // tiles are x[token_of_row[row]] ([T, D] bf16, D = n_out1), copied by the
    // gather warps; the full barriers then also count their arrivals
    const __nv_bfloat16 *xg;
    int x_rows;           // gather: T (a token id outside [0, T) reads as a zero row)
    const int *token_of_row, *row_of;
    const float *topk_w;
    int k;
    void *out1;           // fp16 y [rows, D]
    int *done;            // SCHED_BOTH: [max_blocks] GEMM1 epilogue warps finished, per block
    int max_blocks;       // SCHED_BOTH: entries of done[]
    int *finish;          // SCHED_BOTH: CTAs finished; the last one zeroes done[] and itself
    int *status;
};

size_t pair_smem_bytes(int E_local) {
    return 1024 + (size_t)P_STAGES * P_STAGE_BYTES + P_XBUF_BYTES + P_YSTAGE_BYTES +
           P_NBARS * sizeof(uint64_t) + 16 +
           sizeof(int) * (4 * (size_t)E_local + 1);
}

// Epilogue warps that signal each finished GEMM1 tile: 4 per CTA, 2 CTAs.
constexpr int P_SIGNALS_PER_TILE = 2 * P_EPI_WARPS;

struct PairTile {
    int mode;                      // 0: GEMM1 tile, 1: GEMM2 tile
    int blk;                       // 256-row block (pair m-tile) index
    int expert, row0, nvalid, nt;  // row0 / nvalid: the pair's first row and valid rows (<= 256)
};

// Tile `v` of the launch's static order: block-major, N tiles inner; under
// SCHED_BOTH the MB * nt0 GEMM1 tiles come first.
__device__ __forceinline__ PairTile decode_pair(int v, const PairParams &p, int MB,
                                                const int *s_mtoff, const int *s_base,
                                                const int *s_valid) {
    PairTile c;
    c.mode = p.sched == SCHED_BOTH ? (v >= MB * p.nt0 ? 1 : 0) : p.sched;
    if (p.sched == SCHED_BOTH && c.mode == 1) v -= MB * p.nt0;
    const int n = c.mode ? p.nt1 : p.nt0;
    c.blk = v / n;
    c.nt = v - c.blk * n;
    c.expert = tile_expert(s_mtoff, p.E_local, c.blk);
    const int lm = c.blk - s_mtoff[c.expert];
    c.row0 = s_base[c.expert] + lm * P_PAIR_M;
    c.nvalid = min(P_PAIR_M, s_valid[c.expert] - lm * P_PAIR_M);
    return c;
}

// SiLU(g) = g / (1 + e^-g) with the fast approximate division (2 ulp in
// fp32, far below h's bf16 rounding).  The correctly rounded division cost
// the e4m3 GEMM1 a third of its time on GB300 (fine-grained GEMM1 alone:
// 221 against 149 us); the bf16 GEMM1, bound by its operands, is unchanged.
// For g < -87 the divisor overflows and the quotient is 0, as SiLU is there.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.f + __expf(-g)); }

// Slot weight of row r of token t (0 when the row is not one of t's slots).
__device__ __forceinline__ float slot_weight(const PairParams &p, int r, int t) {
    if (t < 0) return 0.f;
    const int *ro = p.row_of + (size_t)t * p.k;
    for (int j = 0; j < p.k; ++j)
        if (ro[j] == r) return p.topk_w[(size_t)t * p.k + j];
    return 0.f;
}

__device__ __forceinline__ uint32_t pack_bf16x2_p(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <bool kGather>
__global__ void __launch_bounds__(pair_threads(kGather), 1)
grouped_pair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmX64,
                    const __grid_constant__ CUtensorMap tmX16,
                    const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW3,
                    const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmH64,
                    const __grid_constant__ CUtensorMap tmH16,
                    const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmY,
                    const PairParams p) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    // Every role below assumes a cluster of two CTAs (pair MMAs, the peer's
    // barriers, paired TMEM allocation).  A launch in any other shape does no
    // work and reports it instead of reaching an instruction it cannot run.
    if (cluster_nctarank() != 2) {
        if (threadIdx.x == 0) raise_flag(p.status, FLAG_LAUNCH);
        return;
    }
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    // transposed GEMM1 tiles hand the up values over through xbuf [2][32 tokens][32 lanes]
    float *xbuf = reinterpret_cast<float *>(ring + P_STAGES * P_STAGE_BYTES);
    uint8_t *ystage = ring + P_STAGES * P_STAGE_BYTES + P_XBUF_BYTES;  // 1 KB aligned
    uint64_t *bars =
        reinterpret_cast<uint64_t *>(ring + P_STAGES * P_STAGE_BYTES + P_XBUF_BYTES + P_YSTAGE_BYTES);
    uint64_t *full = bars;                   // [P_STAGES]  leader: both CTAs' TMA -> MMA
    uint64_t *empty = bars + P_STAGES;       // [P_STAGES]  MMA -> each CTA's TMA
    uint64_t *tfull = bars + 2 * P_STAGES;   // [2]         MMA -> each CTA's epilogue
    uint64_t *tempty = tfull + 2;            // [2]         leader: both epilogues -> MMA
    uint64_t *drain = tempty + 2;            // [1]         leader: MMA completion at exit
    uint64_t *xfull = drain + 1;             // [2]         up warp -> gate warp (transposed GEMM1)
    uint64_t *xempty = xfull + 2;            // [2]         gate warp -> up warp
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + P_NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *last_cta = reinterpret_cast<int *>(tmem_slot + 2);
    int *s_base = reinterpret_cast<int *>(tmem_slot + 4);
    int *s_valid = s_base + p.E_local;
    int *s_end = s_valid + p.E_local;
    int *s_mtoff = s_end + p.E_local;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

    if (warp == 0) {
        build_tile_table(lane, p.E_local, p.e_first, p.rows_alloc, P_PAIR_M, p.seg_off, p.tpe,
                         s_base, s_valid, s_mtoff, blockIdx.x == 0 ? p.status : nullptr, s_end);
        if (lane == 0) {
            for (int s = 0; s < P_STAGES; ++s) {
                // the leader's producer posts both CTAs' bytes (and, gathering, the
                // stage's gather warp in each CTA arrives once its rows are stored)
                mbar_init(&full[s], kGather ? 1 + 2 : 1);
                mbar_init(&empty[s], 1);   // one multicast commit per use
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(&tfull[a], 1);
                mbar_init(&tempty[a], P_SIGNALS_PER_TILE);  // epilogue warps of both CTAs
            }
            mbar_init(drain, 1);
            for (int a = 0; a < 2; ++a) {
                mbar_init(&xfull[a], 1);
                mbar_init(&xempty[a], 1);
            }
            *abort_flag = 0;
            fence_mbarrier_init();
            if (p.sched != SCHED_GEMM2) {
                prefetch_tmap(&tmX);
                prefetch_tmap(&tmX64);
                prefetch_tmap(&tmX16);
                prefetch_tmap(&tmW1);
                prefetch_tmap(&tmW3);
            }
            if (p.sched != SCHED_GEMM1) {
                prefetch_tmap(&tmY);
                prefetch_tmap(&tmH);
                prefetch_tmap(&tmH64);
                prefetch_tmap(&tmH16);
                prefetch_tmap(&tmW2);
            }
        }
    } else if (warp == 1) {
        tmem_alloc_pair(tmem_slot, P_TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers exist before anything arrives on them
    tc_fence_after();

    const uint32_t tmem_base = *tmem_slot;
    int n_blocks = s_mtoff[p.E_local];
    if (p.sched == SCHED_BOTH && n_blocks > p.max_blocks) {
        // only inconsistent (overlapping) segments get here: nothing is computed
        if (threadIdx.x == 0) raise_flag(p.status, FLAG_BAD_ROUTING);
        n_blocks = 0;
    }
    const int total_tiles =
        n_blocks * (p.sched == SCHED_GEMM1 ? p.nt0 : p.sched == SCHED_GEMM2 ? p.nt1 : p.nt0 + p.nt1);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            const uint32_t full_leader = mapa_shared(smem_u32(&full[0]), 0);
            int s = 0;
            uint32_t ph = 0;
            for (int tile = pair_id; tile < total_tiles; tile += n_pairs) {
                const PairTile c = decode_pair(tile, p, n_blocks, s_mtoff, s_base, s_valid);
                const bool swap = c.nvalid <= P_SWAP_MAX;         // transposed tail tile
                const bool half = !swap && c.nvalid <= P_BM;      // M=128: 64 rows per CTA
                const int srows = ((c.nvalid + 31) & ~31) / 2;    // transposed: token rows per CTA
                const int arow = c.row0 + (int)rank * (swap ? srows : half ? P_BM / 2 : P_BM);
                // gathering: the token rows of GEMM1 tiles come from the gather warps
                const bool gath = kGather && c.mode == 0;
                const uint32_t tx =
                    2u * (swap ? P_A_BYTES + (gath ? 0 : srows * P_BK * 2)
                               : (gath ? 0 : half ? P_A_BYTES / 2 : P_A_BYTES) + P_B_BYTES);
                const CUtensorMap *ta = c.mode ? (half ? &tmH64 : &tmH) : (half ? &tmX64 : &tmX);
                const CUtensorMap *t16 = c.mode ? &tmH16 : &tmX16;
                const int nk = c.mode ? p.nk1 : p.nk0;
                // K elements per stage: 64 bf16 or 128 e4m3 (128 bytes either way)
                const int kel = (c.mode == 0 && p.g1_fp8) ? 2 * P_BK : P_BK;
                bool ok = true;
                if (c.mode == 1 && p.sched == SCHED_BOTH) {
                    // h rows of this block: every GEMM1 tile of the block has stored them
                    if (!wait_count_bounded(p.done + c.blk, P_SIGNALS_PER_TILE * p.nt0, abort_flag))
                        break;
                    fence_proxy_async_global();
                }
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
                    if (leader) {
                        mbar_arrive_expect_tx(&full[s], tx);
                        // a GEMM2 stage has no gathered rows: their arrivals are posted here
                        if (kGather && c.mode != 0) mbar_arrive_cnt(&full[s], 2);
                    }
                    uint8_t *sa = ring + s * P_STAGE_BYTES;
                    uint8_t *sb = sa + P_A_BYTES;
                    const uint32_t fb = full_leader + (uint32_t)(s * sizeof(uint64_t));
                    if (swap) {
                        // weights into the A slot (this CTA's 128 of the 256 M rows),
                        // token rows into the B slot (this CTA's half of N), 16 rows a load
                        if (c.mode == 0) {
                            const int hrow = c.nt * 128 + (int)rank * 64;
                            tma_load_3d_pair(sa, &tmW1, fb, kb * kel, hrow, c.expert);
                            tma_load_3d_pair(sa + P_A_BYTES / 2, &tmW3, fb, kb * kel, hrow, c.expert);
                        } else {
                            tma_load_3d_pair(sa, &tmW2, fb, kb * P_BK, c.nt * P_BN + (int)rank * 128,
                                             c.expert);
                        }
                        if (!gath)
                            for (int i = 0; i < srows / 16; ++i)
                                tma_load_2d_pair(sb + i * 16 * P_BK * 2, t16, fb, kb * kel,
                                                 arow + 16 * i);
                        if (++s == P_STAGES) { s = 0; ph ^= 1u; }
                        continue;
                    }
                    if (!gath) tma_load_2d_pair(sa, ta, fb, kb * kel, arow);
                    if (c.mode == 0) {
                        const int hrow = c.nt * 128 + (int)rank * 64;
                        tma_load_3d_pair(sb, &tmW1, fb, kb * kel, hrow, c.expert);
                        tma_load_3d_pair(sb + P_B_BYTES / 2, &tmW3, fb, kb * kel, hrow, c.expert);
                    } else {
                        tma_load_3d_pair(sb, &tmW2, fb, kb * P_BK, c.nt * P_BN + (int)rank * 128,
                                         c.expert);
                    }
                    if (++s == P_STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (leader CTA) ----------------
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            int it = 0;
            for (int tile = pair_id; ok && tile < total_tiles; tile += n_pairs, ++it) {
                const int acc = it & 1;
                const uint32_t acc_ph = (uint32_t)(it >> 1) & 1u;
                const PairTile c = decode_pair(tile, p, n_blocks, s_mtoff, s_base, s_valid);
                const bool f8 = c.mode == 0 && p.g1_fp8;
                const int mm = c.nvalid <= P_BM && c.nvalid > P_SWAP_MAX ? P_PAIR_M / 2 : P_PAIR_M;
                const int nn = c.nvalid <= P_SWAP_MAX ? (c.nvalid + 31) & ~31 : P_BN;
                const uint32_t idesc = f8 ? idesc_e4m3_f32(mm, nn) : idesc_bf16_f32(mm, nn);
                const int nk = c.mode ? p.nk1 : p.nk0;
                if (!mbar_wait_bounded(&tempty[acc], acc_ph ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * P_ACC_COLS);
                for (int kb = 0; kb < nk; ++kb) {
                    // gathered rows of the peer were written by its threads: cluster acquire
                    if (!mbar_wait_bounded(&full[s], ph, abort_flag, kGather && MOE_GATHER_ACQ_CLUSTER)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(ring + s * P_STAGE_BYTES);
                    const uint32_t b_addr = a_addr + P_A_BYTES;
                    // four MMAs of 32 bytes of K each: K = 16 bf16 or 32 e4m3
                    if (f8) {
#pragma unroll
                        for (int kk = 0; kk < P_BK / 16; ++kk)
                            tc_mma_f8_pair(d_tmem, sdesc_kmajor_sw128(a_addr + kk * 32),
                                           sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                                           (kb | kk) != 0 ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < P_BK / 16; ++kk)
                            tc_mma_f16_pair(d_tmem, sdesc_kmajor_sw128(a_addr + kk * 32),
                                            sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                                            (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit_pair(&empty[s], 0x3);
                    if (++s == P_STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                tc_commit_pair(&tfull[acc], 0x3);
            }
            // every MMA issued here completes before either CTA frees TMEM
            tc_commit_pair(drain, 0x1);
            volatile int local_abort = 0;
            mbar_wait_bounded(drain, 0u, &local_abort);
        }
    } else if (warp < 2 + P_EPI_WARPS) {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        // Each warp owns 32 accumulator rows (its TMEM lane quarter).  h
        // (GEMM1) goes out straight from registers, valid rows only.  GEMM2's
        // y, rounded to fp16, goes out through a swizzled smem box and a TMA
        // store per 64 columns (double-buffered) when all 32 of the warp's rows
        // are valid, else straight from registers as well, so rows without a
        // token are never written.
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        uint8_t *ybuf = ystage + (warp - 2) * 2 * P_YBOX_BYTES;
        uint32_t n_ystore = 0;  // TMA stores issued by this warp (selects the box)
        const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty[0]), 0);
        int it = 0;
        uint32_t xi = 0;  // handoffs done through xbuf (transposed GEMM1 tiles)
        bool xok = true;
        for (int tile = pair_id; xok && tile < total_tiles; tile += n_pairs, ++it) {
            const PairTile c = decode_pair(tile, p, n_blocks, s_mtoff, s_base, s_valid);
            const int acc = it & 1;
            const uint32_t acc_ph = (uint32_t)(it >> 1) & 1u;
            const bool got = mbar_wait_bounded(&tfull[acc], acc_ph, abort_flag);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            if (c.nvalid <= P_SWAP_MAX) {
                // Transposed tile: TMEM lane l holds weight row l of this CTA's
                // 128 and columns 0..nsw-1 hold the tile's tokens.
                const int nsw = (c.nvalid + 31) & ~31;
                const int l = q * 32 + lane;
                const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * P_ACC_COLS);
                if (c.mode == 1) {
                    // y column of this lane; each store is 32 consecutive fp16 of one row
                    const int dcol = c.nt * P_BN + (int)rank * 128 + l;
                    __half *ycol = static_cast<__half *>(p.out1) + (size_t)c.row0 * p.n_out1 + dcol;
                    bool over = false;  // a stored value beyond the fp16 range
#pragma unroll 1
                    for (int ch = 0; ch < nsw / 32; ++ch) {
                        uint32_t d[32];
                        tmem_ld_32x32b_x32(tb + ch * 32, d);
                        // fused combine: lane j looks up token ch * 32 + j and its
                        // slot weight; the warp takes them by shuffle
                        int tl = -1;
                        float wl = 0.f;
                        if (p.comb && ch * 32 + lane < c.nvalid) {
                            const int rr = c.row0 + ch * 32 + lane;
                            tl = p.token_of_row[rr];
                            wl = slot_weight(p, rr, tl);
                        }
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int tj = p.comb ? __shfl_sync(0xffffffffu, tl, j) : -1;
                            const float wj = p.comb ? __shfl_sync(0xffffffffu, wl, j) : 0.f;
                            if (dcol < p.n_out1 && ch * 32 + j < c.nvalid) {
                                if (!p.comb) {
                                    const float v = __uint_as_float(d[j]);
                                    over |= fabsf(v) >= kHalfOverflow;
                                    ycol[(size_t)(ch * 32 + j) * p.n_out1] = __float2half_rn(v);
                                } else if (tj >= 0)
                                    atomicAdd(p.comb + (size_t)tj * p.n_out1 + dcol,
                                              wj * __uint_as_float(d[j]));
                            }
                        }
                    }
                    if (__any_sync(0xffffffffu, over) && lane == 0) raise_flag(p.status, FLAG_RANGE);
                } else {
                    // lanes 0-63: gate of hidden unit u, lanes 64-127: up of the same
                    // units.  The up warps (quarters 2, 3) hand their values to the
                    // gate warps (quarters 0, 1) through xbuf, one 32-token chunk at a
                    // time; the gate warps write h.
                    const int slot = q & 1;
                    float *xb = xbuf + slot * 1024;  // [32 tokens][32 lanes]
                    const int u = c.nt * 128 + (int)rank * 64 + (l & 63);
                    __nv_bfloat16 *hcol = static_cast<__nv_bfloat16 *>(p.out0) + (size_t)c.row0 * p.n_out0 + u;
                    // FP8 GEMM1: this lane's hidden unit's w1 / w3 scales
                    const bool scaled = p.g1_fp8 && q < 2 && u < p.n_out0;
                    const float sw1u = scaled ? p.w1_scale[(size_t)c.expert * p.n_out0 + u] : 1.f;
                    const float sw3u = scaled ? p.w3_scale[(size_t)c.expert * p.n_out0 + u] : 1.f;
#pragma unroll 1
                    for (int ch = 0; ch < nsw / 32; ++ch, ++xi) {
                        uint32_t d[32];
                        tmem_ld_32x32b_x32(tb + ch * 32, d);
                        tc_wait_ld();
                        const uint32_t xph = xi & 1u;
                        if (q >= 2) {
                            const bool ok = mbar_wait_bounded(&xempty[slot], xph ^ 1u, abort_flag);
                            if (!__all_sync(0xffffffffu, ok)) { xok = false; break; }
#pragma unroll
                            for (int j = 0; j < 32; ++j) xb[j * 32 + lane] = __uint_as_float(d[j]);
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&xfull[slot]);
                        } else {
                            const bool ok = mbar_wait_bounded(&xfull[slot], xph, abort_flag);
                            if (!__all_sync(0xffffffffu, ok)) { xok = false; break; }
                            // FP8: lane j fetches the x scale of token ch * 32 + j and
                            // the whole warp takes it by shuffle (uniform control flow)
                            const bool f8s = p.g1_fp8 != 0;
                            const float sxl = f8s && ch * 32 + lane < c.nvalid
                                                  ? p.x_scale[c.row0 + ch * 32 + lane] : 1.f;
                            {
#pragma unroll
                                for (int j = 0; j < 32; ++j) {
                                    const float sx = f8s ? __shfl_sync(0xffffffffu, sxl, j) : 1.f;
                                    if (u < p.n_out0 && ch * 32 + j < c.nvalid) {
                                        float gv = __uint_as_float(d[j]);
                                        float uv = xb[j * 32 + lane];
                                        if (scaled) {
                                            gv *= sx * sw1u;
                                            uv *= sx * sw3u;
                                        }
                                        hcol[(size_t)(ch * 32 + j) * p.n_out0] =
                                            __float2bfloat16_rn(silu_f(gv) * uv);
                                        if (p.gu_out) {
                                            __nv_bfloat16 *gr = p.gu_out +
                                                (size_t)(c.row0 + ch * 32 + j) * 2 * p.n_out0 + u;
                                            gr[0] = __float2bfloat16_rn(gv);
                                            gr[p.n_out0] = __float2bfloat16_rn(uv);
                                        }
                                    }
                                }
                            }
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&xempty[slot]);
                        }
                    }
                    if (!xok) break;
                }
            } else {
            // Rows and columns this lane drains.  Full tile: lane l holds row l
            // and the pair's N columns 0..255.  Half tile: lane l holds row
            // l % 64 and N columns 128*(l / 64) .. +127 in TMEM columns 0..127.
            const bool half = c.nvalid <= P_BM;
            const int rows_cta = half ? P_BM / 2 : P_BM;
            const int crow0 = c.row0 + (int)rank * rows_cta;                // this CTA's rows
            const int cvalid = max(0, min(rows_cta, c.nvalid - (int)rank * rows_cta));
            const int l = q * 32 + lane;
            const int r = half ? (l & 63) : l;
            const int nhalf = half ? (l >> 6) : 0;                          // N half of this lane
            const bool row_ok = r < cvalid;
            const bool warp_has_rows = (half ? (q & 1) * 32 : q * 32) < cvalid;
            const int n_out = c.mode ? p.n_out1 : p.n_out0;
            const size_t orow = (size_t)(crow0 + (row_ok ? r : 0)) * n_out;
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * P_ACC_COLS);
            if (warp_has_rows) {
                if (c.mode == 0) {
                    // h chunks of 32 hidden units: gate at TMEM column gc, up at gc + 64
                    __nv_bfloat16 *hrow = static_cast<__nv_bfloat16 *>(p.out0) + orow;
                    const int nch = half ? 2 : 4;
                    // FP8 GEMM1: the row's x scale; column scales of w1 / w3 below
                    const float sxr = p.g1_fp8 && row_ok ? p.x_scale[crow0 + r] : 1.f;
                    const float *sw1 = p.g1_fp8 ? p.w1_scale + (size_t)c.expert * p.n_out0 : nullptr;
                    const float *sw3 = p.g1_fp8 ? p.w3_scale + (size_t)c.expert * p.n_out0 : nullptr;
#pragma unroll 1
                    for (int ch = 0; ch < nch; ++ch) {
                        const int gc = half ? ch * 32 : (ch >> 1) * 128 + (ch & 1) * 32;
                        const int hcol = half ? nhalf * 64 + ch * 32 : ch * 32;
                        const int col0 = c.nt * 128 + hcol;
                        // FP8: lane i fetches the scales of unit col0 + i (in flight
                        // with the TMEM loads); the elements take them by shuffle
                        float s1 = 1.f, s3 = 1.f;
                        if (p.g1_fp8 && col0 + lane < n_out) {
                            s1 = sw1[col0 + lane];
                            s3 = sw3[col0 + lane];
                        }
                        uint32_t g[32], u[32];
                        tmem_ld_32x32b_x32(tbase + gc, g);
                        tmem_ld_32x32b_x32(tbase + gc + 64, u);
                        tc_wait_ld();
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            if (col0 + v * 8 >= n_out) break;  // uniform across the warp
                            // FP8: row scale times the units' scales, shuffled from
                            // the lanes that fetched them (every lane takes part)
                            float a1[8], a3[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                a1[i] = p.g1_fp8 ? sxr * __shfl_sync(0xffffffffu, s1, v * 8 + i) : 1.f;
                                a3[i] = p.g1_fp8 ? sxr * __shfl_sync(0xffffffffu, s3, v * 8 + i) : 1.f;
                            }
                            if (!row_ok) continue;
                            uint32_t w[4];
#pragma unroll
                            for (int e2 = 0; e2 < 4; ++e2) {
                                float hv[2];
#pragma unroll
                                for (int z = 0; z < 2; ++z) {
                                    const int idx = v * 8 + e2 * 2 + z;
                                    float gv = __uint_as_float(g[idx]);
                                    float uv = __uint_as_float(u[idx]);
                                    if (p.g1_fp8) {
                                        gv *= a1[e2 * 2 + z];
                                        uv *= a3[e2 * 2 + z];
                                    }
                                    hv[z] = silu_f(gv) * uv;
                                }
                                w[e2] = pack_bf16x2_p(hv[0], hv[1]);
                            }
                            *reinterpret_cast<uint4 *>(hrow + col0 + v * 8) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                            if (p.gu_out) {
                                // training forward: keep g and u for the backward
                                __nv_bfloat16 *gr = p.gu_out +
                                    (size_t)(crow0 + r) * 2 * p.n_out0 + col0 + v * 8;
                                uint32_t pg[4], pu[4];
#pragma unroll
                                for (int e2 = 0; e2 < 4; ++e2) {
                                    pg[e2] = pack_bf16x2_p(__uint_as_float(g[v * 8 + e2 * 2]),
                                                           __uint_as_float(g[v * 8 + e2 * 2 + 1]));
                                    pu[e2] = pack_bf16x2_p(__uint_as_float(u[v * 8 + e2 * 2]),
                                                           __uint_as_float(u[v * 8 + e2 * 2 + 1]));
                                }
                                *reinterpret_cast<uint4 *>(gr) = make_uint4(pg[0], pg[1], pg[2], pg[3]);
                                *reinterpret_cast<uint4 *>(gr + p.n_out0) =
                                    make_uint4(pu[0], pu[1], pu[2], pu[3]);
                            }
                        }
                    }
                } else {
                    // y in fp16: two 32-column TMEM chunks make one 128-byte row of 64 values
                    __half *yrow = static_cast<__half *>(p.out1) + orow;
                    const int nch = half ? 4 : P_BN / 32;
                    // this warp's 32 rows start at wrow within the CTA's rows
                    const int wrow = half ? (q & 1) * 32 : q * 32;
                    const bool tma_y = MOE_PAIR_TMA_Y && !p.comb && wrow + 32 <= cvalid;
                    // fused combine: this lane's token and slot weight
                    int tok = -1;
                    float wr = 0.f;
                    if (p.comb && row_ok) {
                        tok = p.token_of_row[crow0 + r];
                        wr = slot_weight(p, crow0 + r, tok);
                    }
                    float *crow = p.comb && tok >= 0 ? p.comb + (size_t)tok * n_out : nullptr;
                    bool over = false;  // a stored value beyond the fp16 range
#pragma unroll 1
                    for (int ch = 0; ch < nch; ch += 2) {
                        uint32_t d[64];
                        tmem_ld_32x32b_x32(tbase + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(d));
                        tmem_ld_32x32b_x32(tbase + (ch + 1) * 32,
                                           *reinterpret_cast<uint32_t(*)[32]>(d + 32));
                        tc_wait_ld();
                        const int col0 = c.nt * P_BN + nhalf * 128 + ch * 32;
                        if (p.comb) {
                            if (row_ok && crow) {
#pragma unroll
                                for (int v = 0; v < 16; ++v) {
                                    if (col0 + v * 4 >= n_out) break;
                                    atomicAdd(reinterpret_cast<float4 *>(crow + col0 + v * 4),
                                              make_float4(wr * __uint_as_float(d[v * 4]),
                                                          wr * __uint_as_float(d[v * 4 + 1]),
                                                          wr * __uint_as_float(d[v * 4 + 2]),
                                                          wr * __uint_as_float(d[v * 4 + 3])));
                                }
                            }
                            continue;
                        }
                        uint32_t hv[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float a = __uint_as_float(d[2 * i]), b = __uint_as_float(d[2 * i + 1]);
                            // only values that are stored count: rows without a token
                            // and columns past n_out (n_out is even) hold garbage
                            if (row_ok && col0 + 2 * i < n_out)
                                over |= fabsf(a) >= kHalfOverflow || fabsf(b) >= kHalfOverflow;
                            hv[i] = pack_half2(a, b);
                        }
                        if (tma_y) {
                            if (col0 >= n_out) continue;  // uniform across the warp
                            if (lane == 0) bulk_wait_group_read<1>();  // this box's last store has read it
                            __syncwarp();
                            // row `lane` of the box; 16-byte unit j at (j ^ (lane & 7))
                            uint8_t *brow = ybuf + (n_ystore & 1) * P_YBOX_BYTES + lane * 128;
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                *reinterpret_cast<uint4 *>(brow + ((j ^ (lane & 7)) << 4)) =
                                    make_uint4(hv[j * 4], hv[j * 4 + 1], hv[j * 4 + 2], hv[j * 4 + 3]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d(&tmY, ybuf + (n_ystore & 1) * P_YBOX_BYTES, col0,
                                             crow0 + wrow);
                                bulk_commit_group();
                            }
                            ++n_ystore;
                            continue;
                        }
                        if (row_ok) {
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                if (col0 + v * 8 >= n_out) break;
                                *reinterpret_cast<uint4 *>(yrow + col0 + v * 8) =
                                    make_uint4(hv[v * 4], hv[v * 4 + 1], hv[v * 4 + 2], hv[v * 4 + 3]);
                            }
                        }
                    }
                    if (__any_sync(0xffffffffu, over) && lane == 0) raise_flag(p.status, FLAG_RANGE);
                }
            }
            }
            tc_fence_before();
            if (c.mode == 0 && p.sched == SCHED_BOTH) {
                // publish this warp's h stores to the GEMM2 producers (TMA
                // readers) of the block: every lane orders its own stores
                // for the async proxy
                // (__syncwarp orders the lanes' stores before lane 0's
                // release, which is cumulative; a per-lane __threadfence was
                // measured 1.3% slower on the fine-grained call)
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) red_release_gpu_add(p.done + c.blk, 1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader + (uint32_t)(acc * sizeof(uint64_t)));
        }
    } else if constexpr (kGather) {
        // ---------------- GEMM1 A-row gather (warps 6..9) ----------------
        // Gather warp g fills the pipeline stages n with n % 4 == g, so four
        // stages are in flight across the warps.  For its stage the warp loads
        // every A row of this CTA (the token rows of a transposed tile, which
        // go to the B slot): the row's 128-byte K slice of x[token_of_row[row]],
        // four whole rows per instruction (lanes 8 i .. 8 i + 7: row 4 it + i,
        // 16-byte piece lane & 7), into registers; pad rows and the K tail past
        // D are zeros.  The loads are in flight while the warp waits for the
        // stage to be free.  It then stores the pieces where the 128-byte
        // swizzle of a TMA load puts them (piece j of row r at j ^ (r & 7)),
        // orders the stores for the async proxy (the MMA reads the stage
        // through it) and lane 0 arrives on the leader's full barrier.  The
        // warp has no load outstanding when it fences and arrives, so neither
        // waits for another stage's loads.
        const int gw = warp - 2 - P_EPI_WARPS;
        const int sub = lane >> 3, ch = lane & 7;
        const uint32_t full_leader = mapa_shared(smem_u32(&full[0]), 0);
        const int upr = p.n_out1 / 8;  // 16-byte units in a row of x (D / 8)
        const uint4 *xv = reinterpret_cast<const uint4 *>(p.xg);
        int s = 0;
        uint32_t ph = 0, n = 0;  // ring position, its phase, stages passed
        bool ok = true;
        for (int tile = pair_id; ok && tile < total_tiles; tile += n_pairs) {
            const PairTile c = decode_pair(tile, p, n_blocks, s_mtoff, s_base, s_valid);
            const int nk = c.mode ? p.nk1 : p.nk0;
            if (c.mode != 0) {  // A is h, loaded by TMA; the producer arrives for us
                for (int kb = 0; kb < nk; ++kb, ++n)
                    if (++s == P_STAGES) { s = 0; ph ^= 1u; }
                continue;
            }
            const bool swap = c.nvalid <= P_SWAP_MAX;
            const bool half = !swap && c.nvalid <= P_BM;
            const int nrows = swap ? ((c.nvalid + 31) & ~31) / 2 : half ? P_BM / 2 : P_BM;
            const int rel0 = (int)rank * nrows;  // this CTA's first row within the pair tile
            // lane l holds the tokens of rows l, l + 32, l + 64, l + 96
            int tk[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = q * 32 + lane;
                tk[q] = r < nrows && rel0 + r < c.nvalid ? p.token_of_row[c.row0 + rel0 + r] : -1;
                if (tk[q] >= p.x_rows) tk[q] = -1;
            }
            const int slot = swap ? P_A_BYTES : 0;
            for (int kb = 0; kb < nk; ++kb, ++n) {
                if ((int)(n % P_GATHER_WARPS) == gw) {
                    const int u = kb * (P_BK / 8) + ch;
                    uint4 b[32];
#pragma unroll
                    for (int it = 0; it < 32; ++it) {
                        const int r = it * 4 + sub;
                        const int t = __shfl_sync(0xffffffffu, tk[it >> 3], r & 31);
                        b[it] = make_uint4(0u, 0u, 0u, 0u);
                        if (r < nrows && t >= 0 && u < upr) b[it] = __ldcg(xv + (size_t)t * upr + u);
                    }
                    // lane 0 waits for the free stage and the warp follows it; the
                    // warp stops as a whole if the wait gave up
                    bool got = true;
                    if (lane == 0) got = mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag);
                    if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
                    uint8_t *st = ring + s * P_STAGE_BYTES + slot;
#pragma unroll
                    for (int it = 0; it < 32; ++it) {
                        const int r = it * 4 + sub;
                        if (r < nrows)
                            *reinterpret_cast<uint4 *>(st + r * 128 + ((ch ^ (r & 7)) << 4)) = b[it];
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(full_leader + (uint32_t)(s * sizeof(uint64_t)));
                }
                if (++s == P_STAGES) { s = 0; ph ^= 1u; }
            }
        }
    }

    if (warp >= 2 && warp < 2 + P_EPI_WARPS && (threadIdx.x & 31) == 0)
        bulk_wait_group_all();  // every y store has landed before the CTA exits
    tc_fence_before();
    __syncthreads();
    // after an abort this CTA's producer may have loads in flight for stages
    // the MMA warp never consumed; the peer waits at the cluster barrier too
    if (threadIdx.x == 0 && *abort_flag) settle_inflight_copies();
    cluster_sync();  // the leader's MMAs (which read both CTAs' smem) are done
    if (threadIdx.x == 0 && *abort_flag) {
        raise_flag(p.status, FLAG_TIMEOUT);
        atomicCAS(p.status + 1, 0, 1 + blockIdx.x);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, P_TMEM_COLS);
    }
    if (p.sched == SCHED_BOTH) {
        // every CTA is past its last read of done[]; the last one to get here
        // leaves the counters zero for the next launch on this workspace
        if (threadIdx.x == 0) {
            __threadfence();
            *last_cta = atomicAdd(p.finish, 1) == (int)gridDim.x - 1;
        }
        __syncthreads();
        if (*last_cta) {
            __threadfence();
            for (int i = threadIdx.x; i < n_blocks; i += blockDim.x) p.done[i] = 0;
            if (threadIdx.x == 0) *p.finish = 0;
        }
    }
}

// clusters of two that fit at once on the current device (0 if none)
template <bool G>
int max_pair_clusters_t(size_t smem) {
    constexpr int kMaxDev = 64;
    static int cached[kMaxDev] = {0};
    static size_t cached_smem[kMaxDev] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    if (cached[dev] > 0 && cached_smem[dev] == smem) return cached[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 256);
    cfg.blockDim = dim3(pair_threads(G));
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void *)grouped_pair_kernel<G>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cached[dev] = n;
    cached_smem[dev] = smem;
    return n;
}

int max_pair_clusters(size_t smem, bool gather) {
    const int n = max_pair_clusters_t<false>(smem);
    return gather ? std::min(n, max_pair_clusters_t<true>(smem)) : n;
}

struct PairMaps {
    CUtensorMap x, x64, x16, w1, w3, h, h64, h16, w2, y;
};

cudaError_t launch_pair(const PairMaps &m, const PairParams &p, int clusters, size_t smem,
                        bool cooperative, bool gather, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(pair_threads(gather));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    // the cooperative one-launch form keeps plain stream order; the
    // two-launch form may start while the previous kernel drains
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    if (cooperative) {
        attr[1].id = cudaLaunchAttributeCooperative;
        attr[1].val.cooperative = 1;
    } else {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (cooperative || MOE_PDL) ? 2 : 1;
    const cudaError_t e =
        gather ? cudaLaunchKernelEx(&cfg, grouped_pair_kernel<true>, m.x, m.x64, m.x16, m.w1, m.w3,
                                    m.h, m.h64, m.h16, m.w2, m.y, p)
               : cudaLaunchKernelEx(&cfg, grouped_pair_kernel<false>, m.x, m.x64, m.x16, m.w1, m.w3,
                                    m.h, m.h64, m.h16, m.w2, m.y, p);
    if (e == cudaSuccess) count_launch();
    return e;
}

// 0: not known yet, 1: this device runs cooperative cluster launches, -1: it refused one
int g_coop_ok[64] = {0};

// A CUDA profiler attached to the process: Nsight Compute starts its target
// with NV_NSIGHT_INJECTION_TRANSPORT_TYPE and NV_COMPUTE_PROFILER_PERFWORKS_DIR
// in the environment, CUPTI-based tools name their injection library in
// CUDA_INJECTION64_PATH.  Under Nsight Compute the cooperative cluster launch
// of both GEMMs has ended in LaunchFailed while the same program ran clean
// without it, so with a profiler attached the GEMMs always run as two
// launches of the same kernel (the form the profiles describe).
bool profiler_attached() {
    static const bool attached = [] {
        for (const char *name : {"NV_NSIGHT_INJECTION_TRANSPORT_TYPE",
                                 "NV_COMPUTE_PROFILER_PERFWORKS_DIR", "CUDA_INJECTION64_PATH"}) {
            const char *v = getenv(name);
            if (v != nullptr && v[0] != '\0') return true;
        }
        return false;
    }();
    return attached;
}

}  // namespace

int64_t grouped_pair_scratch_ints(int64_t rows_alloc, int E_local) {
    return 32 + (rows_alloc + P_PAIR_M - 1) / P_PAIR_M + E_local;
}

namespace {

// Runs GEMM1 + GEMM2 of the tile table: one cooperative launch for short
// calls where the device accepts it, else two launches.
cudaError_t run_pair(const PairMaps &m, const PairParams &p, int64_t rows_alloc, int E_local,
                     int clusters_max, size_t smem, int *scratch, cudaStream_t stream,
                     bool *launched, bool gather = false) {
    const long long pt_bound = (rows_alloc + P_PAIR_M - 1) / P_PAIR_M + E_local;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = -1;
    cudaError_t err;
#ifndef MOE_PAIR_FUSED
#define MOE_PAIR_FUSED 1
#endif
    // One launch pays the prologue once and starts GEMM2 under GEMM1's last
    // wave; it wins on short calls (fine-grained, about 28 tiles per cluster:
    // 0.352 vs 0.366 ms) and measured 3% slower on long ones (DeepSeek-V3-
    // shaped, about 174 tiles per cluster: 5.41 vs 5.27 ms; Zipf-skewed, 203:
    // even), so long calls keep two launches.
    const long long tiles_est = pt_bound * (p.nt0 + p.nt1);
    const bool short_call = tiles_est <= 64LL * clusters_max;
    if (MOE_PAIR_FUSED && short_call && scratch && dev >= 0 && g_coop_ok[dev] >= 0 &&
        !profiler_attached()) {
        // one cooperative launch over both GEMMs; scratch[0] = finish count,
        // scratch[32..] = per-block GEMM1 counts (zero between launches)
        PairParams pb = p;
        pb.sched = SCHED_BOTH;
        const int c = (int)std::min<long long>(clusters_max, pt_bound * (p.nt0 + p.nt1));
        pb.finish = scratch;
        pb.done = scratch + 32;
        pb.max_blocks = (int)pt_bound;
        err = launch_pair(m, pb, c, smem, true, gather, stream);
        if (err == cudaSuccess) {
            g_coop_ok[dev] = 1;
            *launched = true;
            return cudaSuccess;
        }
        if (g_coop_ok[dev] == 1) return err;  // worked before: a real launch failure
        cudaGetLastError();                   // refused: remember, use two launches
        g_coop_ok[dev] = -1;
    }

    PairParams p1 = p;
    p1.sched = SCHED_GEMM1;
    const int c1 = (int)std::min<long long>(clusters_max, pt_bound * p.nt0);
    if ((err = launch_pair(m, p1, c1, smem, false, gather, stream)) != cudaSuccess) return err;
    PairParams p2 = p;
    p2.sched = SCHED_GEMM2;  // A is h: the plain instantiation
    const int c2 = (int)std::min<long long>(clusters_max, pt_bound * p.nt1);
    if ((err = launch_pair(m, p2, c2, smem, false, false, stream)) != cudaSuccess) return err;
    *launched = true;
    return cudaSuccess;
}

PairParams pair_params(const int *seg_offsets, const int *tokens_per_expert, void *h,
                       void *y_perm, int D, int H_local, int e_first, int E_local,
                       int64_t rows_alloc, int *status) {
    PairParams p{};
    p.E_local = E_local;
    p.e_first = e_first;
    p.rows_alloc = (int)rows_alloc;
    p.nk0 = (D + P_BK - 1) / P_BK;
    p.nk1 = (H_local + P_BK - 1) / P_BK;
    p.nt0 = (H_local + 127) / 128;
    p.nt1 = (D + P_BN - 1) / P_BN;
    p.n_out0 = H_local;
    p.n_out1 = D;
    p.seg_off = seg_offsets;
    p.tpe = tokens_per_expert;
    p.out0 = h;
    p.out1 = y_perm;
    p.status = status;
    return p;
}

}  // namespace

cudaError_t launch_grouped_swiglu_bf16_pair(const void *x_perm, const int *seg_offsets,
                                            const int *tokens_per_expert, const void *w1,
                                            const void *w3, const void *w2, void *h, void *y_perm,
                                            int D, int H_local, int e_first, int E_local,
                                            int64_t rows_alloc, int *scratch, int *status,
                                            cudaStream_t stream, bool *launched, void *gu,
                                            const FusedCombine *fc, const GatherA *ga) {
    *launched = false;
    if (E_local == 0 || rows_alloc == 0) {
        *launched = true;
        return cudaSuccess;
    }
    const size_t smem = pair_smem_bytes(E_local);
    if (smem > 227 * 1024) return cudaSuccess;  // not launched: caller falls back
    cudaError_t err = ensure_smem((const void *)grouped_pair_kernel<false>, smem);
    if (err != cudaSuccess) return err;
    if (ga && (err = ensure_smem((const void *)grouped_pair_kernel<true>, smem)) != cudaSuccess)
        return err;
    const int clusters_max = max_pair_clusters(smem, ga != nullptr);
    if (clusters_max <= 0) return cudaSuccess;  // not launched: caller falls back

    PairMaps m;
    // gathering, the x maps are not read; they are built over x so they are valid
    const void *xa = ga ? ga->x : x_perm;
    const int64_t xrows = ga ? ga->T : rows_alloc;
    if (!make_tmap_2d(&m.x, xa, D, xrows, P_BM) ||
        !make_tmap_2d(&m.x64, xa, D, xrows, P_BM / 2) ||
        !make_tmap_2d(&m.x16, xa, D, xrows, 16) ||
        !make_tmap_3d(&m.w1, w1, D, H_local, E_local, 64) ||
        !make_tmap_3d(&m.w3, w3, D, H_local, E_local, 64) ||
        !make_tmap_2d(&m.h, h, H_local, rows_alloc, P_BM) ||
        !make_tmap_2d(&m.h64, h, H_local, rows_alloc, P_BM / 2) ||
        !make_tmap_2d(&m.h16, h, H_local, rows_alloc, 16) ||
        !make_tmap_3d(&m.w2, w2, H_local, D, E_local, 128) ||
        !make_tmap_tile(&m.y, y_perm, 2, D, rows_alloc, 0, 64, 32, 128))
        return cudaErrorInvalidValue;
    PairParams p = pair_params(seg_offsets, tokens_per_expert, h, y_perm, D, H_local, e_first,
                               E_local, rows_alloc, status);
    p.gu_out = (__nv_bfloat16 *)gu;
    if (ga) {
        p.xg = (const __nv_bfloat16 *)ga->x;
        p.x_rows = (int)ga->T;
        p.token_of_row = ga->token_of_row;
    }
    if (fc) {
        p.comb = fc->comb;
        p.token_of_row = fc->token_of_row;
        p.row_of = fc->row_of;
        p.topk_w = fc->topk_w;
        p.k = fc->k;
    }
    return run_pair(m, p, rows_alloc, E_local, clusters_max, smem, scratch, stream, launched,
                    ga != nullptr);
}

cudaError_t launch_grouped_swiglu_fp8_pair(const uint8_t *x_perm_q, const float *x_scale,
                                           const int *seg_offsets, const int *tokens_per_expert,
                                           const uint8_t *w1_q, const float *w1_scale,
                                           const uint8_t *w3_q, const float *w3_scale,
                                           const void *w2, void *h, void *y_perm, int D,
                                           int H_local, int e_first, int E_local,
                                           int64_t rows_alloc, int *scratch, int *status,
                                           cudaStream_t stream, bool *launched) {
    *launched = false;
    if (E_local == 0 || rows_alloc == 0) {
        *launched = true;
        return cudaSuccess;
    }
    const size_t smem = pair_smem_bytes(E_local);
    if (smem > 227 * 1024) return cudaSuccess;  // not launched
    cudaError_t err = ensure_smem((const void *)grouped_pair_kernel<false>, smem);
    if (err != cudaSuccess) return err;
    const int clusters_max = max_pair_clusters(smem, false);
    if (clusters_max <= 0) return cudaSuccess;  // not launched

    // e4m3 operands of GEMM1: boxes of 128 K elements (128 bytes, the same
    // 128-byte swizzled rows as the bf16 boxes of 64)
    PairMaps m;
    if (!make_tmap_tile(&m.x, x_perm_q, 1, D, rows_alloc, 0, 128, P_BM, 128) ||
        !make_tmap_tile(&m.x64, x_perm_q, 1, D, rows_alloc, 0, 128, P_BM / 2, 128) ||
        !make_tmap_tile(&m.x16, x_perm_q, 1, D, rows_alloc, 0, 128, 16, 128) ||
        !make_tmap_tile(&m.w1, w1_q, 1, D, H_local, E_local, 128, 64, 128) ||
        !make_tmap_tile(&m.w3, w3_q, 1, D, H_local, E_local, 128, 64, 128) ||
        !make_tmap_2d(&m.h, h, H_local, rows_alloc, P_BM) ||
        !make_tmap_2d(&m.h64, h, H_local, rows_alloc, P_BM / 2) ||
        !make_tmap_2d(&m.h16, h, H_local, rows_alloc, 16) ||
        !make_tmap_3d(&m.w2, w2, H_local, D, E_local, 128) ||
        !make_tmap_tile(&m.y, y_perm, 2, D, rows_alloc, 0, 64, 32, 128))
        return cudaErrorInvalidValue;
    PairParams p = pair_params(seg_offsets, tokens_per_expert, h, y_perm, D, H_local, e_first,
                               E_local, rows_alloc, status);
    p.g1_fp8 = 1;
    p.nk0 = (D + 2 * P_BK - 1) / (2 * P_BK);
    p.x_scale = x_scale;
    p.w1_scale = w1_scale;
    p.w3_scale = w3_scale;
    return run_pair(m, p, rows_alloc, E_local, clusters_max, smem, scratch, stream, launched);
}

}  // namespace moe
