// bf16 m-grouped SwiGLU expert FFN on the 5th-generation tensor cores.
//
// Page "Expert Parallelism (EP)" (llm-infra-atlas), section 1 (routed
// experts compute fc1 -> act -> fc2 as one grouped GEMM over the permuted
// rows) and section 2 (an m-grouped kernel runs same-shaped GEMMs whose M
// differs, a tile scheduler spanning the groups; its input layout is the
// dispatch output: expert-contiguous, M-tile aligned).  Weights in the
// GroupedExperts convention of "Expert Tensor Parallel design", section 4.3:
// w1/w3 [E, H, D], w2 [E, D, H] -- both operands of both GEMMs are K-major.
//
// Kernel design (sm_103a):
//   * persistent: one CTA per SM walks a static list of output tiles
//     (m-tile of one expert x n-tile); the per-expert tile table is built in
//     shared memory from the segment offsets in device memory, so the host
//     never waits for the routing counts;
//   * warp-specialised: warp 0 issues TMA loads into a 4-stage shared-memory
//     ring (mbarrier transaction counts), warp 1 issues tcgen05.mma
//     (M=128, N=256, K=16, bf16 -> fp32) into one of two TMEM accumulators,
//     warps 2-5 drain the other accumulator (tcgen05.ld) and store it;
//   * GEMM1 (mode 0) stacks 128 rows of w1 and the same 128 rows of w3 into
//     one N=256 B tile, so each accumulator holds gate and up for the same
//     hidden units and the epilogue writes h = SiLU(gate) * up directly;
//   * GEMM2 (mode 1) is a plain N=256 tile of w2; its fp32 accumulator is
//     stored as fp16 (11 significant bits; the weighted combine sums in fp32
//     and rounds the token's output to bf16 once).
//   * every mbarrier wait is bounded; a wait that runs out raises
//     FLAG_TIMEOUT, the CTA drains its copies and MMAs, frees TMEM and exits.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int TC_BM = 128, TC_BN = 256, TC_BK = 64, TC_STAGES = 4;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;  // 16 KB
constexpr int TC_B_BYTES = TC_BN * TC_BK * 2;  // 32 KB
constexpr int TC_STAGE_BYTES = TC_A_BYTES + TC_B_BYTES;
constexpr int TC_THREADS = 192;
constexpr int TC_ACC_COLS = 256;
constexpr int TC_TMEM_COLS = 512;
constexpr uint32_t TC_IDESC = idesc_bf16_f32(TC_BM, TC_BN);

struct TcParams {
    int mode;       // 0: h = SiLU(A w1^T) * (A w3^T);  1: y = A w2^T
    int E_local, e_first;
    int K;          // reduction length (D for mode 0, H_local for mode 1)
    int N_out;      // output columns (H_local for mode 0, D for mode 1)
    int n_tiles;    // output tiles along N (128 columns in mode 0, 256 in mode 1)
    int rows_alloc;
    const int *seg_off;
    const int *tpe;
    void *out;      // mode 0: bf16 h [rows, H_local]; mode 1: fp16 y [rows, D]
    int *status;
};

size_t tc_smem_bytes(int E_local) {
    return 1024                                    // alignment slack
           + (size_t)TC_STAGES * TC_STAGE_BYTES    // operand ring
           + 16 * sizeof(uint64_t)                 // barriers
           + 16                                    // tmem slot, abort flag
           + sizeof(int) * (3 * (size_t)E_local + 1);
}

struct TileCoord {
    int expert, row0, nvalid, nt;
};

__device__ __forceinline__ TileCoord decode_tile(int tile, int n_tiles, const int *s_mtoff,
                                                 const int *s_base, const int *s_valid,
                                                 int E_local) {
    TileCoord c;
    const int mt = tile / n_tiles;
    c.nt = tile - mt * n_tiles;
    c.expert = tile_expert(s_mtoff, E_local, mt);
    const int lm = mt - s_mtoff[c.expert];
    c.row0 = s_base[c.expert] + lm * TC_BM;
    c.nvalid = min(TC_BM, s_valid[c.expert] - lm * TC_BM);
    return c;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// A tile with at most TC_A16_MAX valid rows loads only those rows, in boxes
// of 16 (tmA16), instead of the whole 128-row A box; the rows past them hold
// whatever the stage held before and give output rows that are not stored.
// (Masked decode: about four rows per expert, so the full box read 32x the
// needed bytes of x_perm and h.)
constexpr int TC_A16_MAX = 64;

__global__ void __launch_bounds__(TC_THREADS, 1)
grouped_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA16,
                  const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                  const TcParams p) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + TC_STAGES * TC_STAGE_BYTES);
    uint64_t *full = bars;                    // [TC_STAGES]  TMA -> MMA
    uint64_t *empty = bars + TC_STAGES;       // [TC_STAGES]  MMA -> TMA
    uint64_t *tfull = bars + 2 * TC_STAGES;   // [2]          MMA -> epilogue
    uint64_t *tempty = tfull + 2;             // [2]          epilogue -> MMA
    uint64_t *drain = tempty + 2;             // [1]          MMA completion at exit
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_base = reinterpret_cast<int *>(tmem_slot + 4);
    int *s_valid = s_base + p.E_local;
    int *s_mtoff = s_valid + p.E_local;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        build_tile_table(lane, p.E_local, p.e_first, p.rows_alloc, TC_BM, p.seg_off, p.tpe,
                         s_base, s_valid, s_mtoff, blockIdx.x == 0 ? p.status : nullptr);
        if (lane == 0) {
            for (int s = 0; s < TC_STAGES; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], 1);
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(&tfull[a], 1);
                mbar_init(&tempty[a], 4);  // one arrive per epilogue warp
            }
            mbar_init(drain, 1);
            *abort_flag = 0;
            fence_mbarrier_init();
            prefetch_tmap(&tmA);
            prefetch_tmap(&tmA16);
            prefetch_tmap(&tmB0);
            if (p.mode == 0) prefetch_tmap(&tmB1);
        }
    } else if (warp == 1) {
        tmem_alloc(tmem_slot, TC_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_slot;
    const int total_tiles = s_mtoff[p.E_local] * p.n_tiles;
    const int nk = (p.K + TC_BK - 1) / TC_BK;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int s = 0;
            uint32_t ph = 0;
            int last_parity[TC_STAGES];
            for (int q = 0; q < TC_STAGES; ++q) last_parity[q] = -1;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                const TileCoord c = decode_tile(tile, p.n_tiles, s_mtoff, s_base, s_valid, p.E_local);
                const int na16 = c.nvalid <= TC_A16_MAX ? (c.nvalid + 15) / 16 : 0;
                const uint32_t tx = (na16 ? na16 * 16 * TC_BK * 2 : TC_A_BYTES) + TC_B_BYTES;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[s], tx);
                    uint8_t *sa = ring + s * TC_STAGE_BYTES;
                    uint8_t *sb = sa + TC_A_BYTES;
                    if (na16) {
                        for (int i = 0; i < na16; ++i)
                            tma_load_2d(sa + i * 16 * TC_BK * 2, &tmA16, &full[s], kb * TC_BK,
                                        c.row0 + 16 * i);
                    } else {
                        tma_load_2d(sa, &tmA, &full[s], kb * TC_BK, c.row0);
                    }
                    if (p.mode == 0) {
                        tma_load_3d(sb, &tmB0, &full[s], kb * TC_BK, c.nt * 128, c.expert);
                        tma_load_3d(sb + TC_B_BYTES / 2, &tmB1, &full[s], kb * TC_BK, c.nt * 128,
                                    c.expert);
                    } else {
                        tma_load_3d(sb, &tmB0, &full[s], kb * TC_BK, c.nt * TC_BN, c.expert);
                    }
                    last_parity[s] = (int)ph;
                    if (++s == TC_STAGES) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // let every copy already issued land before the CTA exits
                volatile int local_abort = 0;
                for (int q = 0; q < TC_STAGES; ++q)
                    if (last_parity[q] >= 0)
                        mbar_wait_bounded(&full[q], (uint32_t)last_parity[q], &local_abort);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            int it = 0;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t acc_ph = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait_bounded(&tempty[acc], acc_ph ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * TC_ACC_COLS);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait_bounded(&full[s], ph, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(ring + s * TC_STAGE_BYTES);
                    const uint32_t b_addr = a_addr + TC_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < TC_BK / 16; ++kk) {
                        tc_mma_f16(d_tmem, sdesc_kmajor_sw128(a_addr + kk * 32),
                                   sdesc_kmajor_sw128(b_addr + kk * 32), TC_IDESC,
                                   (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(&empty[s]);
                    if (++s == TC_STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                tc_commit(&tfull[acc]);
            }
            // every MMA issued by this thread completes before TMEM is freed
            tc_commit(drain);
            volatile int local_abort = 0;
            mbar_wait_bounded(drain, 0u, &local_abort);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        int it = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
            const TileCoord c = decode_tile(tile, p.n_tiles, s_mtoff, s_base, s_valid, p.E_local);
            const int acc = it & 1;
            const uint32_t acc_ph = (uint32_t)(it >> 1) & 1u;
            // every lane waits; the vote keeps the warp converged for tcgen05.ld
            const bool got = mbar_wait_bounded(&tfull[acc], acc_ph, abort_flag);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            const int r = q * 32 + lane;
            const bool row_ok = r < c.nvalid;
            const size_t orow = (size_t)(c.row0 + (row_ok ? r : 0)) * p.N_out;
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * TC_ACC_COLS);
            if (p.mode == 0) {
                __nv_bfloat16 *hrow = static_cast<__nv_bfloat16 *>(p.out) + orow;
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t g[32], u[32];
                    tmem_ld_32x32b_x32(tbase + ch * 32, g);
                    tmem_ld_32x32b_x32(tbase + 128 + ch * 32, u);
                    tc_wait_ld();
                    const int col0 = c.nt * 128 + ch * 32;
                    if (row_ok) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            if (col0 + v * 8 >= p.N_out) break;
                            uint32_t w[4];
#pragma unroll
                            for (int e2 = 0; e2 < 4; ++e2) {
                                float hv[2];
#pragma unroll
                                for (int z = 0; z < 2; ++z) {
                                    const int idx = v * 8 + e2 * 2 + z;
                                    const float gv = __uint_as_float(g[idx]);
                                    const float uv = __uint_as_float(u[idx]);
                                    hv[z] = gv / (1.f + __expf(-gv)) * uv;
                                }
                                w[e2] = pack_bf16x2(hv[0], hv[1]);
                            }
                            *reinterpret_cast<uint4 *>(hrow + col0 + v * 8) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            } else {
                __half *yrow = static_cast<__half *>(p.out) + orow;
                bool over = false;  // a stored value beyond the fp16 range
#pragma unroll 1
                for (int ch = 0; ch < TC_BN / 32; ++ch) {
                    uint32_t d[32];
                    tmem_ld_32x32b_x32(tbase + ch * 32, d);
                    tc_wait_ld();
                    const int col0 = c.nt * TC_BN + ch * 32;
                    if (row_ok) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            if (col0 + v * 8 >= p.N_out) break;
                            uint32_t w[4];
#pragma unroll
                            for (int e2 = 0; e2 < 4; ++e2) {
                                const float a = __uint_as_float(d[v * 8 + e2 * 2]);
                                const float b = __uint_as_float(d[v * 8 + e2 * 2 + 1]);
                                over |= fabsf(a) >= kHalfOverflow || fabsf(b) >= kHalfOverflow;
                                w[e2] = pack_half2(a, b);
                            }
                            *reinterpret_cast<uint4 *>(yrow + col0 + v * 8) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                if (__any_sync(0xffffffffu, over) && lane == 0) raise_flag(p.status, FLAG_RANGE);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        raise_flag(p.status, FLAG_TIMEOUT);
        atomicCAS(p.status + 1, 0, 1 + blockIdx.x);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TC_TMEM_COLS);
    }
}

// ---------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------
}  // namespace

cudaError_t launch_grouped_swiglu_bf16(const void *x_perm, const int *seg_offsets,
                                       const int *tokens_per_expert, const void *w1,
                                       const void *w3, const void *w2, void *h, void *y_perm,
                                       int D, int H_local, int e_first, int E_local,
                                       int64_t rows_alloc, int *status, cudaStream_t stream) {
    if (E_local == 0 || rows_alloc == 0) return cudaSuccess;
    CUtensorMap tm_x, tm_x16, tm_w1, tm_w3, tm_h, tm_h16, tm_w2;
    if (!make_tmap_2d(&tm_x, x_perm, D, rows_alloc, TC_BM) ||
        !make_tmap_2d(&tm_x16, x_perm, D, rows_alloc, 16) ||
        !make_tmap_3d(&tm_w1, w1, D, H_local, E_local, 128) ||
        !make_tmap_3d(&tm_w3, w3, D, H_local, E_local, 128) ||
        !make_tmap_2d(&tm_h, h, H_local, rows_alloc, TC_BM) ||
        !make_tmap_2d(&tm_h16, h, H_local, rows_alloc, 16) ||
        !make_tmap_3d(&tm_w2, w2, H_local, D, E_local, TC_BN))
        return cudaErrorInvalidValue;
    const int nsm = sm_count();
    if (nsm <= 0) return cudaErrorNoDevice;
    const size_t smem = tc_smem_bytes(E_local);
    cudaError_t err = ensure_smem((const void *)grouped_tc_kernel, smem);
    if (err != cudaSuccess) return err;
    const long long mt_bound = (rows_alloc + TC_BM - 1) / TC_BM + E_local;

    TcParams p1{};
    p1.mode = 0;
    p1.E_local = E_local;
    p1.e_first = e_first;
    p1.K = D;
    p1.N_out = H_local;
    p1.n_tiles = (H_local + 127) / 128;
    p1.rows_alloc = (int)rows_alloc;
    p1.seg_off = seg_offsets;
    p1.tpe = tokens_per_expert;
    p1.out = h;
    p1.status = status;
    const long long g1 = std::min<long long>(nsm, mt_bound * p1.n_tiles);
    if ((err = launch_pdl(grouped_tc_kernel, dim3((unsigned)g1), dim3(TC_THREADS), smem, stream,
                          tm_x, tm_x16, tm_w1, tm_w3, p1)) != cudaSuccess)
        return err;
    count_launch();
    if ((err = cudaGetLastError()) != cudaSuccess) return err;

    TcParams p2 = p1;
    p2.mode = 1;
    p2.K = H_local;
    p2.N_out = D;
    p2.n_tiles = (D + TC_BN - 1) / TC_BN;
    p2.out = y_perm;
    const long long g2 = std::min<long long>(nsm, mt_bound * p2.n_tiles);
    if ((err = launch_pdl(grouped_tc_kernel, dim3((unsigned)g2), dim3(TC_THREADS), smem, stream,
                          tm_h, tm_h16, tm_w2, tm_w2, p2)) != cudaSuccess)
        return err;
    count_launch();
    return cudaGetLastError();
}

}  // namespace moe
