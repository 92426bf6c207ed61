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
//     consecutive 128-row halves of a 256-row w2 tile and store y in fp32;
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
//     cluster barrier before TMEM is freed.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int P_BM = 128;                        // rows per CTA
constexpr int P_PAIR_M = 2 * P_BM;               // rows per pair tile
constexpr int P_BN = 256;                        // N of the pair MMA
constexpr int P_BK = 64;
#ifndef MOE_PAIR_STAGES
#define MOE_PAIR_STAGES 6
#endif
constexpr int P_STAGES = MOE_PAIR_STAGES;
constexpr int P_A_BYTES = P_BM * P_BK * 2;       // 16 KB
constexpr int P_B_BYTES = (P_BN / 2) * P_BK * 2; // 16 KB: this CTA's half of B
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
constexpr int P_THREADS = 192;
constexpr int P_ACC_COLS = 256;
constexpr int P_TMEM_COLS = 512;
constexpr uint32_t P_IDESC = idesc_bf16_f32(P_PAIR_M, P_BN);
constexpr uint32_t P_IDESC_HALF = idesc_bf16_f32(P_PAIR_M / 2, P_BN);
constexpr int P_NBARS = 24;


struct PairParams {
    int mode;       // 0: h = SiLU(A w1^T) * (A w3^T);  1: y = A w2^T
    int E_local, e_first;
    int K;          // reduction length
    int N_out;      // output columns
    int n_tiles;    // output tiles along N (128 columns in mode 0, 256 in mode 1)
    int rows_alloc;
    const int *seg_off;
    const int *tpe;
    void *out;      // mode 0: bf16 h [rows, H_local]; mode 1: fp32 y [rows, D]
    int *status;
};

size_t pair_smem_bytes(int E_local) {
    return 1024 + (size_t)P_STAGES * P_STAGE_BYTES + P_NBARS * sizeof(uint64_t) + 16 +
           sizeof(int) * (4 * (size_t)E_local + 1);
}

struct PairTile {
    int expert, row0, nvalid, nt;  // row0 / nvalid: the pair's first row and valid rows (<= 256)
};

__device__ __forceinline__ PairTile decode_pair(int tile, int n_tiles, const int *s_mtoff,
                                                const int *s_base, const int *s_valid,
                                                int E_local) {
    PairTile c;
    const int mt = tile / n_tiles;
    c.nt = tile - mt * n_tiles;
    c.expert = tile_expert(s_mtoff, E_local, mt);
    const int lm = mt - s_mtoff[c.expert];
    c.row0 = s_base[c.expert] + lm * P_PAIR_M;
    c.nvalid = min(P_PAIR_M, s_valid[c.expert] - lm * P_PAIR_M);
    return c;
}

__device__ __forceinline__ uint32_t pack_bf16x2_p(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(P_THREADS, 1)
grouped_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA64,
                    const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                    const PairParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + P_STAGES * P_STAGE_BYTES);
    uint64_t *full = bars;                   // [P_STAGES]  leader: both CTAs' TMA -> MMA
    uint64_t *empty = bars + P_STAGES;       // [P_STAGES]  MMA -> each CTA's TMA
    uint64_t *tfull = bars + 2 * P_STAGES;   // [2]         MMA -> each CTA's epilogue
    uint64_t *tempty = tfull + 2;            // [2]         leader: both epilogues -> MMA
    uint64_t *drain = tempty + 2;            // [1]         leader: MMA completion at exit
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + P_NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
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
                mbar_init(&full[s], 1);    // the leader's producer posts both CTAs' bytes
                mbar_init(&empty[s], 1);   // one multicast commit per use
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(&tfull[a], 1);
                mbar_init(&tempty[a], 8);  // 4 epilogue warps x 2 CTAs
            }
            mbar_init(drain, 1);
            *abort_flag = 0;
            fence_mbarrier_init();
            prefetch_tmap(&tmA);
            prefetch_tmap(&tmA64);
            prefetch_tmap(&tmB0);
            if (p.mode == 0) prefetch_tmap(&tmB1);
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
    const int total_tiles = s_mtoff[p.E_local] * p.n_tiles;
    const int nk = (p.K + P_BK - 1) / P_BK;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            const uint32_t full_leader = mapa_shared(smem_u32(&full[0]), 0);
            int s = 0;
            uint32_t ph = 0;
            for (int tile = pair_id; tile < total_tiles; tile += n_pairs) {
                const PairTile c = decode_pair(tile, p.n_tiles, s_mtoff, s_base, s_valid, p.E_local);
                const bool half = c.nvalid <= P_BM;  // M=128: 64 rows per CTA
                const int arow = c.row0 + (int)rank * (half ? P_BM / 2 : P_BM);
                const uint32_t tx = 2u * (half ? P_A_BYTES / 2 + P_B_BYTES : P_STAGE_BYTES);
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
                    if (leader) mbar_arrive_expect_tx(&full[s], tx);
                    uint8_t *sa = ring + s * P_STAGE_BYTES;
                    uint8_t *sb = sa + P_A_BYTES;
                    const uint32_t fb = full_leader + (uint32_t)(s * sizeof(uint64_t));
                    tma_load_2d_pair(sa, half ? &tmA64 : &tmA, fb, kb * P_BK, arow);
                    if (p.mode == 0) {
                        const int hrow = c.nt * 128 + (int)rank * 64;
                        tma_load_3d_pair(sb, &tmB0, fb, kb * P_BK, hrow, c.expert);
                        tma_load_3d_pair(sb + P_B_BYTES / 2, &tmB1, fb, kb * P_BK, hrow, c.expert);
                    } else {
                        tma_load_3d_pair(sb, &tmB0, fb, kb * P_BK, c.nt * P_BN + (int)rank * 128,
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
                const PairTile c = decode_pair(tile, p.n_tiles, s_mtoff, s_base, s_valid, p.E_local);
                const uint32_t idesc = c.nvalid <= P_BM ? P_IDESC_HALF : P_IDESC;
                if (!mbar_wait_bounded(&tempty[acc], acc_ph ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * P_ACC_COLS);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait_bounded(&full[s], ph, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(ring + s * P_STAGE_BYTES);
                    const uint32_t b_addr = a_addr + P_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < P_BK / 16; ++kk) {
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
    } else {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        // Each warp owns 32 accumulator rows (its TMEM lane quarter) and
        // stores them straight from registers, valid rows only.  (Staging
        // through shared memory for TMA stores was measured slower: the
        // stores then compete with the operand loads for the TMA unit.)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty[0]), 0);
        int it = 0;
        for (int tile = pair_id; tile < total_tiles; tile += n_pairs, ++it) {
            const PairTile c = decode_pair(tile, p.n_tiles, s_mtoff, s_base, s_valid, p.E_local);
            const int acc = it & 1;
            const uint32_t acc_ph = (uint32_t)(it >> 1) & 1u;
            const bool got = mbar_wait_bounded(&tfull[acc], acc_ph, abort_flag);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
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
            const size_t orow = (size_t)(crow0 + (row_ok ? r : 0)) * p.N_out;
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * P_ACC_COLS);
            if (warp_has_rows) {
                if (p.mode == 0) {
                    // h chunks of 32 hidden units: gate at TMEM column gc, up at gc + 64
                    __nv_bfloat16 *hrow = static_cast<__nv_bfloat16 *>(p.out) + orow;
                    const int nch = half ? 2 : 4;
#pragma unroll 1
                    for (int ch = 0; ch < nch; ++ch) {
                        const int gc = half ? ch * 32 : (ch >> 1) * 128 + (ch & 1) * 32;
                        const int hcol = half ? nhalf * 64 + ch * 32 : ch * 32;
                        uint32_t g[32], u[32];
                        tmem_ld_32x32b_x32(tbase + gc, g);
                        tmem_ld_32x32b_x32(tbase + gc + 64, u);
                        tc_wait_ld();
                        const int col0 = c.nt * 128 + hcol;
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
                                    w[e2] = pack_bf16x2_p(hv[0], hv[1]);
                                }
                                *reinterpret_cast<uint4 *>(hrow + col0 + v * 8) =
                                    make_uint4(w[0], w[1], w[2], w[3]);
                            }
                        }
                    }
                } else {
                    float *yrow = static_cast<float *>(p.out) + orow;
                    const int nch = half ? 4 : P_BN / 32;
#pragma unroll 1
                    for (int ch = 0; ch < nch; ++ch) {
                        uint32_t d[32];
                        tmem_ld_32x32b_x32(tbase + ch * 32, d);
                        tc_wait_ld();
                        const int col0 = c.nt * P_BN + nhalf * 128 + ch * 32;
                        if (row_ok) {
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                if (col0 + v * 4 >= p.N_out) break;
                                *reinterpret_cast<uint4 *>(yrow + col0 + v * 4) =
                                    make_uint4(d[v * 4], d[v * 4 + 1], d[v * 4 + 2], d[v * 4 + 3]);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader + (uint32_t)(acc * sizeof(uint64_t)));
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the leader's MMAs (which read both CTAs' smem) are done
    if (threadIdx.x == 0 && *abort_flag) {
        raise_flag(p.status, FLAG_TIMEOUT);
        atomicCAS(p.status + 1, 0, 1 + blockIdx.x);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, P_TMEM_COLS);
    }
}

// clusters of two that fit at once on the current device (0 if none)
int max_pair_clusters(size_t smem) {
    constexpr int kMaxDev = 64;
    static int cached[kMaxDev] = {0};
    static size_t cached_smem[kMaxDev] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    if (cached[dev] > 0 && cached_smem[dev] == smem) return cached[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 256);
    cfg.blockDim = dim3(P_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void *)grouped_pair_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cached[dev] = n;
    cached_smem[dev] = smem;
    return n;
}

cudaError_t launch_pair(const CUtensorMap &a, const CUtensorMap &a64, const CUtensorMap &b0,
                        const CUtensorMap &b1, const PairParams &p, int clusters, size_t smem,
                        cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(P_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launch();
    return cudaLaunchKernelEx(&cfg, grouped_pair_kernel, a, a64, b0, b1, p);
}

}  // namespace

cudaError_t launch_grouped_swiglu_bf16_pair(const void *x_perm, const int *seg_offsets,
                                            const int *tokens_per_expert, const void *w1,
                                            const void *w3, const void *w2, void *h, void *y_perm,
                                            int D, int H_local, int e_first, int E_local,
                                            int64_t rows_alloc, int *status, cudaStream_t stream,
                                            bool *launched) {
    *launched = false;
    if (E_local == 0 || rows_alloc == 0) {
        *launched = true;
        return cudaSuccess;
    }
    const size_t smem = pair_smem_bytes(E_local);
    if (smem > 227 * 1024) return cudaSuccess;  // not launched: caller falls back
    cudaError_t err = ensure_smem((const void *)grouped_pair_kernel, smem);
    if (err != cudaSuccess) return err;
    const int clusters_max = max_pair_clusters(smem);
    if (clusters_max <= 0) return cudaSuccess;  // not launched: caller falls back

    CUtensorMap tm_x, tm_x64, tm_w1, tm_w3, tm_h, tm_h64, tm_w2;
    if (!make_tmap_2d(&tm_x, x_perm, D, rows_alloc, P_BM) ||
        !make_tmap_2d(&tm_x64, x_perm, D, rows_alloc, P_BM / 2) ||
        !make_tmap_3d(&tm_w1, w1, D, H_local, E_local, 64) ||
        !make_tmap_3d(&tm_w3, w3, D, H_local, E_local, 64) ||
        !make_tmap_2d(&tm_h, h, H_local, rows_alloc, P_BM) ||
        !make_tmap_2d(&tm_h64, h, H_local, rows_alloc, P_BM / 2) ||
        !make_tmap_3d(&tm_w2, w2, H_local, D, E_local, 128))
        return cudaErrorInvalidValue;
    const long long pt_bound = (rows_alloc + P_PAIR_M - 1) / P_PAIR_M + E_local;

    PairParams p1{};
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
    const int c1 = (int)std::min<long long>(clusters_max, pt_bound * p1.n_tiles);
    if ((err = launch_pair(tm_x, tm_x64, tm_w1, tm_w3, p1, c1, smem, stream)) != cudaSuccess) return err;

    PairParams p2 = p1;
    p2.mode = 1;
    p2.K = H_local;
    p2.N_out = D;
    p2.n_tiles = (D + P_BN - 1) / P_BN;
    p2.out = y_perm;
    const int c2 = (int)std::min<long long>(clusters_max, pt_bound * p2.n_tiles);
    if ((err = launch_pair(tm_h, tm_h64, tm_w2, tm_w2, p2, c2, smem, stream)) != cudaSuccess) return err;
    *launched = true;
    return cudaSuccess;
}

}  // namespace moe
