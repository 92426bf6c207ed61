// Backward of the grouped SwiGLU experts on CTA pairs (tcgen05 cta_group::2).
//
// Page "Expert Parallelism (EP)" (llm-infra-atlas), section 5: the backward
// mirrors the forward -- the expert weights get m-grouped dgrad GEMMs over
// the same expert-contiguous layout and k-grouped wgrad GEMMs whose reduction
// runs over each expert's rows.  With gy = dL/dy_perm (bf16), g and u the
// forward's gate / up pre-activations (saved as gu [rows, 2H]), per expert e:
//   dh   = gy_e . w2_e                  m-grouped, K = D   (w2_e [D, H]: B MN-major)
//   dg   = dh * u * SiLU'(g),  du = dh * SiLU(g)       fused into dh's epilogue
//   dxp  = [dg | du] . [w1_e ; w3_e]    m-grouped, K = 2H  (w1_e, w3_e [H, D]: B MN-major)
//   dw2_e = gy_e^T . h_e                k-grouped, K = rows of e (both operands MN-major)
//   [dw1_e ; dw3_e] = [dg | du]_e^T . x_e            k-grouped, K = rows of e
// The operands are read in the layouts the forward already has: tcgen05
// reads an MN-major operand straight from shared memory (transpose bits of
// the instruction descriptor), so nothing is transposed in memory.
//
// Structure as the forward pair kernel: a cluster of two CTAs computes a
// 256 x 256 tile with M=256 MMAs, each CTA holding 128 M rows of A and 128
// N columns of B; warp 0 issues TMA into a 6-stage ring of 32 KB, warp 1 of
// the leader issues the MMAs into one of two TMEM accumulators, warps 2-5 of
// both CTAs drain them.  Every wait is bounded (FLAG_TIMEOUT).
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int B_BM = 128;                         // M rows per CTA
constexpr int B_PAIR_M = 2 * B_BM;
constexpr int B_BN = 256;                         // N of the pair MMA
constexpr int B_BK = 64;
constexpr int B_MAX_STAGES = 6;
constexpr int B_A_BYTES = B_BM * B_BK * 2;        // 16 KB
constexpr int B_B_BYTES = (B_BN / 2) * B_BK * 2;  // 16 KB: this CTA's half of B
constexpr int B_STAGE_BYTES = B_A_BYTES + B_B_BYTES;
constexpr int B_CHUNK = 64 * B_BK * 2;            // one MN-major box: 64 M/N elements x 64 K rows
constexpr int B_MAX_EPI_WARPS = 8;  // 4 or 8: each TMEM lane quarter drained by 1 or 2 warps
constexpr int B_MAX_THREADS = 64 + 32 * B_MAX_EPI_WARPS;
constexpr int B_ACC_COLS = 256;
constexpr int B_TMEM_COLS = 512;
constexpr int B_NBARS = 40;
#ifndef MOE_BWD_EPI_WARPS_STORE
#define MOE_BWD_EPI_WARPS_STORE 8
#endif
#ifndef MOE_BWD_EPI_WARPS_SWIGLU
#define MOE_BWD_EPI_WARPS_SWIGLU 4
#endif
#ifndef MOE_BWD_EPI_WARPS_DGRAD
#define MOE_BWD_EPI_WARPS_DGRAD 4
#endif
// Epilogue staging, per epilogue warp: two 4 KB output boxes (32 rows x 32
// fp32, or the dg and du halves of 32 rows x 32 bf16 each) and, for the
// SwiGLU backward, two 4 KB input boxes (the saved g and u of the chunk).
constexpr int B_BOX_BYTES = 4096;
constexpr int B_EPI_BYTES_STORE = 2 * B_BOX_BYTES;
constexpr int B_EPI_BYTES_SWIGLU = 4 * B_BOX_BYTES;

enum : int {
    BS_MGROUPED = 0,  // tiles over each expert's rows; K fixed
    BS_KGROUPED = 1,  // tiles over a per-expert [M, N] output; K = the expert's rows
};
enum : int {
    BE_STORE = 0,        // fp32 store
    BE_SWIGLU_BWD = 1,   // dh -> dg, du (bf16) with the saved g, u
};

struct BwdParams {
    int sched, epi;
    int a_mn, b_mn;        // operand major-ness (1: MN-major)
    int E_local, e_first, rows_alloc;
    int M, N, nk;          // k-grouped: per-expert M x N; m-grouped: N and K / 64
    int mt, nt;            // tiles along M (k-grouped) and N
    int k_split;           // m-grouped: k-blocks >= k_split read B from tmB1 (at k - k_split)
    int m_split;           // k-grouped: output rows m >= m_split go through the second output map
    int stages;            // smem ring depth
    int epi_bytes;         // staging bytes per epilogue warp
    int epi_warps;         // 4 or 8 epilogue warps
    int out_bf16;          // BE_STORE: the output boxes hold bf16 (32 x 32, 64-byte swizzle)
    const int *seg_off, *tpe;
    int H;
    int *status;
};

// Shared memory: 1 KB alignment slack, the ring, the epilogue staging, the
// barriers, the TMEM slot / abort flag and the tile table.
size_t bwd_smem_bytes(int E_local, int stages, int epi_bytes, int epi_warps) {
    return 1024 + (size_t)stages * B_STAGE_BYTES + (size_t)epi_warps * epi_bytes +
           B_NBARS * sizeof(uint64_t) + 16 + sizeof(int) * (4 * (size_t)E_local + 1);
}

// The deepest ring (at most B_MAX_STAGES, at least 2) that fits 227 KB.
int bwd_stages(int E_local, int epi_bytes, int epi_warps) {
    for (int st = B_MAX_STAGES; st >= 2; --st)
        if (bwd_smem_bytes(E_local, st, epi_bytes, epi_warps) <= 227 * 1024) return st;
    return 0;
}

struct BwdTile {
    int expert;
    int row0, nvalid, seg_rows;  // m-grouped: first row, valid rows (<= 256), rows to the segment end
    int m0, n0;                  // k-grouped: output origin; m-grouped: n0
    int kbase, nk;               // first K row (k-grouped) and k-blocks
};

__device__ __forceinline__ BwdTile decode_bwd(int v, const BwdParams &p, const int *s_mtoff,
                                              const int *s_base, const int *s_valid,
                                              const int *s_end) {
    BwdTile c;
    if (p.sched == BS_MGROUPED) {
        const int blk = v / p.nt;
        const int ni = v - blk * p.nt;
        c.expert = tile_expert(s_mtoff, p.E_local, blk);
        const int lm = blk - s_mtoff[c.expert];
        c.row0 = s_base[c.expert] + lm * B_PAIR_M;
        c.nvalid = min(B_PAIR_M, s_valid[c.expert] - lm * B_PAIR_M);
        c.seg_rows = min(B_PAIR_M, s_end[c.expert] - c.row0);
        c.m0 = 0;
        c.n0 = ni * B_BN;
        c.kbase = 0;
        c.nk = p.nk;
    } else {
        const int per = p.mt * p.nt;
        c.expert = v / per;
        const int rem = v - c.expert * per;
        const int mi = rem / p.nt;
        c.m0 = mi * B_PAIR_M;
        c.n0 = (rem - mi * p.nt) * B_BN;
        c.row0 = 0;
        c.nvalid = 0;
        c.seg_rows = 0;
        c.kbase = s_base[c.expert];
        c.nk = (s_valid[c.expert] + B_BK - 1) / B_BK;
    }
    return c;
}

__global__ void __launch_bounds__(B_MAX_THREADS, 1)
bwd_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmO0,
                const __grid_constant__ CUtensorMap tmO1, const BwdParams p) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const int n_st = p.stages;
    uint8_t *epi = ring + n_st * B_STAGE_BYTES;  // 1 KB aligned
    uint64_t *bars = reinterpret_cast<uint64_t *>(epi + p.epi_warps * p.epi_bytes);
    uint64_t *full = bars;                       // [stages] leader: both CTAs' TMA -> MMA
    uint64_t *empty = bars + B_MAX_STAGES;       // [stages] MMA -> each CTA's TMA
    uint64_t *tfull = bars + 2 * B_MAX_STAGES;   // [2]      MMA -> each CTA's epilogue
    uint64_t *tempty = tfull + 2;                // [2]      leader: both epilogues -> MMA
    uint64_t *drain = tempty + 2;                // [1]      leader: MMA completion at exit
    uint64_t *ldbar = drain + 1;                 // [2 per epilogue warp] g/u box loads
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + B_NBARS);
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
        build_tile_table(lane, p.E_local, p.e_first, p.rows_alloc, B_PAIR_M, p.seg_off, p.tpe,
                         s_base, s_valid, s_mtoff, blockIdx.x == 0 ? p.status : nullptr, s_end);
        if (lane == 0) {
            for (int s = 0; s < n_st; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], 1);
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(&tfull[a], 1);
                mbar_init(&tempty[a], 2 * p.epi_warps);  // every epilogue warp of both CTAs
            }
            mbar_init(drain, 1);
            for (int i = 0; i < 2 * p.epi_warps; ++i) mbar_init(&ldbar[i], 1);
            *abort_flag = 0;
            fence_mbarrier_init();
            prefetch_tmap(&tmA);
            prefetch_tmap(&tmB0);
            prefetch_tmap(&tmB1);
            prefetch_tmap(&tmO0);
            prefetch_tmap(&tmO1);
        }
    } else if (warp == 1) {
        tmem_alloc_pair(tmem_slot, B_TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers exist before anything arrives on them
    tc_fence_after();

    const uint32_t tmem_base = *tmem_slot;
    const int total_tiles =
        p.sched == BS_MGROUPED ? s_mtoff[p.E_local] * p.nt : p.E_local * p.mt * p.nt;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            const uint32_t full_leader = mapa_shared(smem_u32(&full[0]), 0);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int tile = pair_id; ok && tile < total_tiles; tile += n_pairs) {
                const BwdTile c = decode_bwd(tile, p, s_mtoff, s_base, s_valid, s_end);
                for (int kb = 0; kb < c.nk; ++kb) {
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
                    if (leader) mbar_arrive_expect_tx(&full[s], 2u * B_STAGE_BYTES);
                    uint8_t *sa = ring + s * B_STAGE_BYTES;
                    uint8_t *sb = sa + B_A_BYTES;
                    const uint32_t fb = full_leader + (uint32_t)(s * sizeof(uint64_t));
                    const int k0 = c.kbase + kb * B_BK;
                    // A: this CTA's 128 M rows
                    if (p.a_mn) {
                        const int m = c.m0 + (int)rank * B_BM;
                        tma_load_2d_pair(sa, &tmA, fb, m, k0);
                        tma_load_2d_pair(sa + B_CHUNK, &tmA, fb, m + 64, k0);
                    } else {
                        tma_load_2d_pair(sa, &tmA, fb, k0, c.row0 + (int)rank * B_BM);
                    }
                    // B: this CTA's 128 N columns, MN-major
                    const int n = c.n0 + (int)rank * (B_BN / 2);
                    if (p.sched == BS_MGROUPED) {
                        const bool hi = kb >= p.k_split;
                        const CUtensorMap *tb = hi ? &tmB1 : &tmB0;
                        const int kk = hi ? (kb - p.k_split) * B_BK : k0;
                        tma_load_3d_pair(sb, tb, fb, n, kk, c.expert);
                        tma_load_3d_pair(sb + B_CHUNK, tb, fb, n + 64, kk, c.expert);
                    } else {
                        tma_load_2d_pair(sb, &tmB0, fb, n, k0);
                        tma_load_2d_pair(sb + B_CHUNK, &tmB0, fb, n + 64, k0);
                    }
                    if (++s == n_st) { s = 0; ph ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (leader CTA) ----------------
            const uint32_t idesc = idesc_bf16_f32_major(B_PAIR_M, B_BN, p.a_mn, p.b_mn);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            int it = 0;
            for (int tile = pair_id; ok && tile < total_tiles; tile += n_pairs, ++it) {
                const int acc = it & 1;
                const uint32_t acc_ph = (uint32_t)(it >> 1) & 1u;
                const BwdTile c = decode_bwd(tile, p, s_mtoff, s_base, s_valid, s_end);
                if (!mbar_wait_bounded(&tempty[acc], acc_ph ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * B_ACC_COLS);
                for (int kb = 0; kb < c.nk; ++kb) {
                    if (!mbar_wait_bounded(&full[s], ph, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(ring + s * B_STAGE_BYTES);
                    const uint32_t b_addr = a_addr + B_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < B_BK / 16; ++kk) {
                        const uint64_t da = p.a_mn ? sdesc_mnmajor_sw128(a_addr + kk * 2048, B_CHUNK)
                                                   : sdesc_kmajor_sw128(a_addr + kk * 32);
                        const uint64_t db = sdesc_mnmajor_sw128(b_addr + kk * 2048, B_CHUNK);
                        tc_mma_f16_pair(d_tmem, da, db, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit_pair(&empty[s], 0x3);
                    if (++s == n_st) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                // an expert without rows issues no MMA: its epilogue writes zeros
                tc_commit_pair(&tfull[acc], 0x3);
            }
            tc_commit_pair(drain, 0x1);
            volatile int local_abort = 0;
            mbar_wait_bounded(drain, 0u, &local_abort);
        }
    } else {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        // Each warp owns 32 accumulator rows (its TMEM lane quarter) and
        // moves them out in 32-column chunks: TMEM -> registers -> a
        // swizzled smem box -> one TMA store, double-buffered so a store
        // drains while the next chunk is formed.  The SwiGLU backward also
        // brings the chunk's saved g and u in by TMA, one chunk ahead.
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int wi = warp - 2;
        // with 8 warps, two share a lane quarter and split the tile's columns
        const int n_grp = p.epi_warps / 4, grp = wi / 4, ch_per = (B_BN / 32) / n_grp;
        uint8_t *stg = epi + wi * p.epi_bytes;   // out boxes [0, 8 KB), in boxes [8, 16 KB)
        uint64_t *lb = ldbar + 2 * wi;
        const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty[0]), 0);
        const bool swiglu = p.epi == BE_SWIGLU_BWD;
        uint32_t n_store = 0, n_load = 0, n_used = 0;  // warp-uniform counters
        bool ok = true;
        int it = 0;
        for (int tile = pair_id; ok && tile < total_tiles; tile += n_pairs, ++it) {
            const BwdTile c = decode_bwd(tile, p, s_mtoff, s_base, s_valid, s_end);
            const int acc = it & 1;
            const uint32_t acc_ph = (uint32_t)(it >> 1) & 1u;
            const int wrow = (int)rank * B_BM + q * 32;  // this warp's first row in the pair tile
            bool active;
            int y0 = 0;  // the box's row coordinate
            const CUtensorMap *to = &tmO0;
            if (p.sched == BS_MGROUPED) {
                active = wrow < c.seg_rows;  // segments end on 32-row boundaries
                y0 = c.row0 + wrow;
            } else {
                const int m = c.m0 + wrow;
                active = m < p.M;
                if (m < p.m_split) {
                    y0 = m;
                } else {
                    y0 = m - p.m_split;
                    to = &tmO1;
                }
            }
            // this warp's chunks: [ch_lo, ch_hi) of the tile's 32-column chunks
            const int ch_lo = grp * ch_per;
            const int ch_hi = active ? min(ch_lo + ch_per, (p.N - c.n0) / 32) : 0;
            const int n_ch = max(0, ch_hi - ch_lo);
            auto issue_load = [&](int ch) {  // g and u of chunk ch -> in box (n_load & 1)
                if (lane == 0) {
                    uint8_t *ib = stg + 2 * B_BOX_BYTES + (n_load & 1) * B_BOX_BYTES;
                    uint64_t *bar = &lb[n_load & 1];
                    const int col = c.n0 + ch * 32;
                    mbar_arrive_expect_tx(bar, B_BOX_BYTES);
                    tma_load_2d(ib, &tmO0, bar, col, y0);
                    tma_load_2d(ib + B_BOX_BYTES / 2, &tmO0, bar, p.H + col, y0);
                }
                ++n_load;
            };
            if (swiglu && n_ch > 0) {
                // the tile's g and u head for L2 while its MMAs run; chunk 0 for smem
                if (lane < 2 * n_ch)
                    tma_prefetch_l2_2d(&tmO0, (lane & 1 ? p.H : 0) + c.n0 + (ch_lo + (lane >> 1)) * 32,
                                       y0);
                issue_load(ch_lo);
            }
            const bool got = mbar_wait_bounded(&tfull[acc], acc_ph, abort_flag);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * B_ACC_COLS);
            const int rl = wrow + lane;  // this lane's row within the pair tile
            const bool valid = rl < c.nvalid;
            const bool empty_expert = p.sched == BS_KGROUPED && c.nk == 0;
#pragma unroll 1
            for (int ch = ch_lo; ch < ch_hi; ++ch) {
                uint32_t d[32];
                tmem_ld_32x32b_x32(tbase + ch * 32, d);
                const uint8_t *ib = nullptr;
                if (swiglu) {
                    if (ch + 1 < ch_hi) issue_load(ch + 1);
                    const bool in_ok =
                        mbar_wait_bounded(&lb[n_used & 1], (n_used >> 1) & 1u, abort_flag);
                    ib = stg + 2 * B_BOX_BYTES + (n_used & 1) * B_BOX_BYTES;
                    ++n_used;
                    if (!__all_sync(0xffffffffu, in_ok)) { ok = false; break; }
                }
                tc_wait_ld();
                if (lane == 0) bulk_wait_group_read<1>();  // this out box's previous store has read it
                __syncwarp();
                uint8_t *ob = stg + (n_store & 1) * B_BOX_BYTES;
                const int col0 = c.n0 + ch * 32;
                if (!swiglu && p.out_bf16) {
                    // 32 x 32 bf16 box, 64-byte swizzle: 16-byte unit j of row r at (j ^ ((r >> 1) & 3))
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t w[4];
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(
                                empty_expert ? 0.f : __uint_as_float(d[j * 8 + e2 * 2]),
                                empty_expert ? 0.f : __uint_as_float(d[j * 8 + e2 * 2 + 1]));
                            w[e2] = *reinterpret_cast<uint32_t *>(&b2);
                        }
                        *reinterpret_cast<uint4 *>(ob + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else if (!swiglu) {
                    // 32 x 32 fp32 box, 128-byte swizzle: 16-byte unit j of row r at (j ^ (r & 7))
                    uint8_t *row = ob + lane * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint4 v = empty_expert ? make_uint4(0, 0, 0, 0)
                                                     : make_uint4(d[j * 4], d[j * 4 + 1],
                                                                  d[j * 4 + 2], d[j * 4 + 3]);
                        *reinterpret_cast<uint4 *>(row + ((j ^ (lane & 7)) << 4)) = v;
                    }
                } else {
                    // g, u in and dg, du out: 32 x 32 bf16 boxes, 64-byte swizzle: 16-byte unit
                    // j of row r at (j ^ ((r >> 1) & 3)); dh -> dg = dh u s (1 + g (1 - s)),
                    // du = dh g s (s the sigmoid of g); rows past the valid ones get zeros
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int off = lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4);
                        const uint4 gq = *reinterpret_cast<const uint4 *>(ib + off);
                        const uint4 uq = *reinterpret_cast<const uint4 *>(ib + B_BOX_BYTES / 2 + off);
                        const __nv_bfloat16 *gv = reinterpret_cast<const __nv_bfloat16 *>(&gq);
                        const __nv_bfloat16 *uv = reinterpret_cast<const __nv_bfloat16 *>(&uq);
                        uint32_t og[4], ou[4];
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            float dg[2], du[2];
#pragma unroll
                            for (int z = 0; z < 2; ++z) {
                                const float dh = __uint_as_float(d[j * 8 + e2 * 2 + z]);
                                const float g = __bfloat162float(gv[e2 * 2 + z]);
                                const float u = __bfloat162float(uv[e2 * 2 + z]);
                                const float sg = __fdividef(1.f, 1.f + __expf(-g));
                                dg[z] = valid ? dh * u * sg * (1.f + g * (1.f - sg)) : 0.f;
                                du[z] = valid ? dh * g * sg : 0.f;
                            }
                            __nv_bfloat162 pg = __floats2bfloat162_rn(dg[0], dg[1]);
                            __nv_bfloat162 pu = __floats2bfloat162_rn(du[0], du[1]);
                            og[e2] = *reinterpret_cast<uint32_t *>(&pg);
                            ou[e2] = *reinterpret_cast<uint32_t *>(&pu);
                        }
                        *reinterpret_cast<uint4 *>(ob + off) = make_uint4(og[0], og[1], og[2], og[3]);
                        *reinterpret_cast<uint4 *>(ob + B_BOX_BYTES / 2 + off) =
                            make_uint4(ou[0], ou[1], ou[2], ou[3]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (swiglu) {
                        tma_store_2d(&tmO1, ob, col0, y0);
                        tma_store_2d(&tmO1, ob + B_BOX_BYTES / 2, p.H + col0, y0);
                    } else if (p.sched == BS_MGROUPED) {
                        tma_store_2d(to, ob, col0, y0);
                    } else {
                        tma_store_3d(to, ob, col0, y0, c.expert);
                    }
                    bulk_commit_group();
                }
                ++n_store;
            }
            if (!ok) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader + (uint32_t)(acc * sizeof(uint64_t)));
        }
        if (lane == 0) bulk_wait_group_all();  // every store has landed before the CTA exits
        // a g/u load still in flight after an abort lands before the smem goes away
        while (n_used < n_load) {
            volatile int local_abort = 0;
            mbar_wait_bounded(&lb[n_used & 1], (n_used >> 1) & 1u, &local_abort);
            ++n_used;
        }
    }

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
        tmem_dealloc_pair(tmem_base, B_TMEM_COLS);
    }
}

int max_bwd_clusters(size_t smem, int threads) {
    constexpr int kMaxDev = 64;
    static int cached[kMaxDev] = {0};
    static size_t cached_smem[kMaxDev] = {0};
    static int cached_threads[kMaxDev] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    if (cached[dev] > 0 && cached_smem[dev] == smem && cached_threads[dev] == threads)
        return cached[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 256);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void *)bwd_pair_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cached[dev] = n;
    cached_smem[dev] = smem;
    cached_threads[dev] = threads;
    return n;
}

cudaError_t launch_bwd(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1,
                       const CUtensorMap &o0, const CUtensorMap &o1, BwdParams p, long long tiles,
                       cudaStream_t stream) {
    p.stages = bwd_stages(p.E_local, p.epi_bytes, p.epi_warps);
    if (p.stages == 0) return cudaErrorInvalidConfiguration;
    const size_t smem = bwd_smem_bytes(p.E_local, p.stages, p.epi_bytes, p.epi_warps);
    const int threads = 64 + 32 * p.epi_warps;
    cudaError_t err = ensure_smem((const void *)bwd_pair_kernel, smem);
    if (err != cudaSuccess) return err;
    const int clusters_max = max_bwd_clusters(smem, threads);
    if (clusters_max <= 0) return cudaErrorLaunchOutOfResources;
    const int clusters = (int)std::max<long long>(1, std::min<long long>(clusters_max, tiles));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = MOE_PDL ? 2 : 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, bwd_pair_kernel, a, b0, b1, o0, o1, p);
    if (e == cudaSuccess) count_launch();
    return e;
}

// The rows that the k-grouped weight gradients read past a segment's valid
// rows -- [b + v, b + ceil64(v)) for local expert i with b = seg_off[i] and v
// its valid rows -- are set to zero in each listed bf16 buffer, so whole
// 64-row K blocks of a segment can be reduced over.  Block (i, y) takes
// every gridDim.y-th such row of expert i.
__global__ void __launch_bounds__(256)
zero_pad_rows_kernel(const int *__restrict__ seg_off, const int *__restrict__ tpe, int e_first,
                     int64_t rows, __nv_bfloat16 *b0, int c0, __nv_bfloat16 *b1, int c1,
                     __nv_bfloat16 *b2, int c2) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    const int i = blockIdx.x;
    const int sb = seg_off[i], se = seg_off[i + 1];
    const int c = tpe[e_first + i];
    if (sb < 0 || se < sb || se > rows || c < 0) return;  // flagged by the GEMM kernels
    const int v = min(c, se - sb);
    const int pad_end = min(se, sb + (v + 63) / 64 * 64);
    const uint4 z = make_uint4(0, 0, 0, 0);
    __nv_bfloat16 *bufs[3] = {b0, b1, b2};
    const int cols[3] = {c0, c1, c2};
    for (int r = sb + v + (int)blockIdx.y; r < pad_end; r += (int)gridDim.y)
        for (int q = 0; q < 3; ++q) {
            if (!bufs[q]) continue;
            uint4 *row = reinterpret_cast<uint4 *>(bufs[q] + (size_t)r * cols[q]);
            for (int u = threadIdx.x; u < cols[q] / 8; u += blockDim.x) row[u] = z;
        }
}

}  // namespace

int64_t grouped_bwd_smem(int E_local) {
    // the largest of the four launches' needs, each with a ring of >= 2 stages
    const int64_t a = (int64_t)bwd_smem_bytes(E_local, 2, B_EPI_BYTES_SWIGLU, MOE_BWD_EPI_WARPS_SWIGLU);
    const int64_t b = (int64_t)bwd_smem_bytes(E_local, 2, B_EPI_BYTES_STORE, MOE_BWD_EPI_WARPS_STORE);
    const int64_t c = (int64_t)bwd_smem_bytes(E_local, 2, B_EPI_BYTES_STORE, MOE_BWD_EPI_WARPS_DGRAD);
    return std::max({a, b, c});
}

cudaError_t launch_grouped_swiglu_bwd(const void *x_perm, const void *h, const void *gu,
                                      const void *gy, const int *seg_offsets,
                                      const int *tokens_per_expert, const int *token_of_row,
                                      const void *w1, const void *w3, const void *w2,
                                      void *dgu, float *dxp, void *dw1, void *dw3, void *dw2,
                                      int D, int H_local, int e_first, int E_local,
                                      int64_t rows_alloc, int *status, cudaStream_t stream,
                                      int grad_bf16) {
    (void)token_of_row;
    if (E_local == 0 || rows_alloc == 0) return cudaSuccess;
    if (D % 32 || H_local % 32) return cudaErrorInvalidValue;  // whole 32-column boxes
    cudaError_t err;
    // padding rows of the saved x_perm and h and of gy read as zeros
    if ((err = launch_pdl(zero_pad_rows_kernel, dim3((unsigned)E_local, 8), dim3(256), 0, stream,
                          seg_offsets, tokens_per_expert, e_first, rows_alloc,
                          (__nv_bfloat16 *)x_perm, D, (__nv_bfloat16 *)h, H_local,
                          (__nv_bfloat16 *)gy, D)) != cudaSuccess)
        return err;
    count_launch();
    const long long blk_bound = (rows_alloc + B_PAIR_M - 1) / B_PAIR_M + E_local;
    const uint64_t rows = (uint64_t)rows_alloc, H2 = 2 * (uint64_t)H_local;

    BwdParams base{};
    base.E_local = E_local;
    base.e_first = e_first;
    base.rows_alloc = (int)rows_alloc;
    base.seg_off = seg_offsets;
    base.tpe = tokens_per_expert;
    base.status = status;
    base.H = H_local;
    base.epi_bytes = B_EPI_BYTES_STORE;
    base.epi_warps = MOE_BWD_EPI_WARPS_STORE;

    CUtensorMap tA, tB0, tB1, tO0, tO1;
    // 1. dh = gy . w2_e, fused SwiGLU backward -> dgu  (m-grouped, K = D)
    {
        BwdParams p = base;
        p.sched = BS_MGROUPED;
        p.epi = BE_SWIGLU_BWD;
        p.epi_bytes = B_EPI_BYTES_SWIGLU;
        p.epi_warps = MOE_BWD_EPI_WARPS_SWIGLU;
        p.a_mn = 0;
        p.b_mn = 1;
        p.N = H_local;
        p.nk = D / B_BK;
        p.nt = (H_local + B_BN - 1) / B_BN;
        p.k_split = p.nk;
        if (!make_tmap_2d(&tA, gy, D, rows_alloc, B_BM) ||
            !make_tmap_3d(&tB0, w2, H_local, D, E_local, B_BK) ||
            !make_tmap_tile(&tO0, gu, 2, H2, rows, 0, 32, 32, 64) ||
            !make_tmap_tile(&tO1, dgu, 2, H2, rows, 0, 32, 32, 64))
            return cudaErrorInvalidValue;
        if ((err = launch_bwd(tA, tB0, tB0, tO0, tO1, p, blk_bound * p.nt, stream)) != cudaSuccess)
            return err;
    }
    // 2. dxp = [dg | du] . [w1_e ; w3_e]  (m-grouped, K = 2H, fp32 out)
    {
        BwdParams p = base;
        p.sched = BS_MGROUPED;
        p.epi = BE_STORE;
        p.a_mn = 0;
        p.b_mn = 1;
        p.N = D;
        p.nk = 2 * H_local / B_BK;
        p.nt = (D + B_BN - 1) / B_BN;
        p.k_split = H_local / B_BK;
        p.epi_warps = MOE_BWD_EPI_WARPS_DGRAD;
        if (!make_tmap_2d(&tA, dgu, H2, rows_alloc, B_BM) ||
            !make_tmap_3d(&tB0, w1, D, H_local, E_local, B_BK) ||
            !make_tmap_3d(&tB1, w3, D, H_local, E_local, B_BK) ||
            !make_tmap_tile(&tO0, dxp, 4, D, rows, 0, 32, 32, 128))
            return cudaErrorInvalidValue;
        if ((err = launch_bwd(tA, tB0, tB1, tO0, tO0, p, blk_bound * p.nt, stream)) != cudaSuccess)
            return err;
    }
    // 3. dw2_e = gy_e^T . h_e  (k-grouped: M = D, N = H)
    {
        BwdParams p = base;
        p.sched = BS_KGROUPED;
        p.epi = BE_STORE;
        p.a_mn = 1;
        p.b_mn = 1;
        p.M = D;
        p.N = H_local;
        p.mt = (D + B_PAIR_M - 1) / B_PAIR_M;
        p.nt = (H_local + B_BN - 1) / B_BN;
        p.m_split = D;
        p.out_bf16 = grad_bf16;
        const int eb = grad_bf16 ? 2 : 4;  // 32-column boxes: 64 or 128 bytes wide
        if (!make_tmap_2d(&tA, gy, D, rows_alloc, B_BK) ||
            !make_tmap_2d(&tB0, h, H_local, rows_alloc, B_BK) ||
            !make_tmap_tile(&tO0, dw2, eb, H_local, D, E_local, 32, 32, 32 * eb))
            return cudaErrorInvalidValue;
        if ((err = launch_bwd(tA, tB0, tB0, tO0, tO0, p, (long long)E_local * p.mt * p.nt,
                              stream)) != cudaSuccess)
            return err;
    }
    // 4. [dw1_e ; dw3_e] = [dg | du]_e^T . x_e  (k-grouped: M = 2H, N = D)
    {
        BwdParams p = base;
        p.sched = BS_KGROUPED;
        p.epi = BE_STORE;
        p.a_mn = 1;
        p.b_mn = 1;
        p.M = 2 * H_local;
        p.N = D;
        p.mt = (2 * H_local + B_PAIR_M - 1) / B_PAIR_M;
        p.nt = (D + B_BN - 1) / B_BN;
        p.m_split = H_local;
        p.out_bf16 = grad_bf16;
        const int eb = grad_bf16 ? 2 : 4;
        if (!make_tmap_2d(&tA, dgu, H2, rows_alloc, B_BK) ||
            !make_tmap_2d(&tB0, x_perm, D, rows_alloc, B_BK) ||
            !make_tmap_tile(&tO0, dw1, eb, D, H_local, E_local, 32, 32, 32 * eb) ||
            !make_tmap_tile(&tO1, dw3, eb, D, H_local, E_local, 32, 32, 32 * eb))
            return cudaErrorInvalidValue;
        if ((err = launch_bwd(tA, tB0, tB0, tO0, tO1, p, (long long)E_local * p.mt * p.nt,
                              stream)) != cudaSuccess)
            return err;
    }
    return cudaSuccess;
}

}  // namespace moe
