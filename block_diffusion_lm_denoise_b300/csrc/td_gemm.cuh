// td_gemm.cuh -- persistent tcgen05 GEMM  C[M, N] = A[M, K] * B[N, K]^T  (bf16 in, fp32
// accumulate in TMEM) with four fused epilogues:
//   EPI_QKV    : bf16 store of the [q | k | v] projection into three row-major tensors
//   EPI_QKV_ROPE: the same with q and k rotated first (rotary positional variant)
//   EPI_RESID  : gated residual  h[r, n] = bf16(h[r, n] + gate[n] * C[r, n])  (in place, or
//                for the last layer of a step only the rows the LM head needs, compacted)
//   EPI_LMHEAD : per row and per 128/256-column vocabulary tile, (max, lowest argmax,
//                sum of exp(z - max)) of the logits; the logits are never written.
//
// Roles (256 threads): warp 0 lane 0 = TMA producer; warp 1 = TMEM allocator and (lane 0)
// MMA issuer; warps 4..7 = epilogue, thread i of warp 4+q owns accumulator row 32q+i.
// Tiles: BM = 128 rows, BN = 128 or 256 columns, BK = 64 (one 128-byte swizzle row of bf16),
// STAGES-deep TMA ring in shared memory, two TMEM accumulators so the epilogue of tile i
// overlaps the MMAs of tile i+1. Work items are (m_tile, n_tile) pairs enumerated with
// m_tile fastest and dealt round-robin to the CTAs, so the CTAs resident at any moment share
// a narrow window of B tiles (the weights) and every weight byte leaves HBM about once.
// gemm_pair_kernel (below) runs the same epilogues on 256 x 256 tiles over SM pairs; the
// library uses it for every 256-wide GEMM and this kernel with BN = 128 for few rows.
// The QKV and residual epilogues store 64-column chunks through an 8 x 8 transpose within
// each lane octet, so that one store instruction writes whole 128-byte rows; the residual
// epilogue reads the gate slice from a per-warp copy in shared memory.
#pragma once

#include "td_ptx.cuh"

namespace td {

enum { EPI_QKV = 0, EPI_RESID = 1, EPI_LMHEAD = 2, EPI_QKV_ROPE = 3 };

struct GemmParams {
  int M, N, K;
  int m_tiles, n_tiles, items;
  // EPI_QKV: columns [0, nq) -> q, [nq, nq + nk) -> k, [nq + nk, nq + 2 nk) -> v; with
  // rope_cs set, q and k are rotated before rounding: row r, pair j of a head (columns 2j,
  // 2j + 1) by rope_cs[r * head_dim / 2 + j] = (cos, sin)
  uint16_t* q;
  uint16_t* k;
  uint16_t* v;
  int nq, nk;
  const float2* rope_cs;
  int head_dim;
  // EPI_RESID; with row_pos set, row r's result goes to row row_pos[r] of h_out instead of
  // back into h, and rows with row_pos[r] < 0 are not written
  uint16_t* h;
  const float* gate;
  const int* row_pos;
  uint16_t* h_out;
  // EPI_LMHEAD partials, [M][n_tiles] each
  float* part_max;
  int* part_arg;
  float* part_sum;
  // when non-null and nonzero, the kernel returns at once (a finished decode loop)
  const int* skip;
  // when non-null: only the first *m_count rows of A are live (read on the device; M is the
  // row capacity of A and of the partials)
  const int* m_count;
};

template <int BN, int STAGES>
struct GemmSmem {
  static constexpr int kABytes = 128 * 128;      // 128 rows x 64 bf16
  static constexpr int kBBytes = BN * 128;       // BN rows x 64 bf16
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOffset = STAGES * kStageBytes;
  static constexpr int kGateOffset = kBarOffset + 256;     // gate slices (EPI_RESID), 4 warps
  static constexpr int kBytes = kGateOffset + 4 * BN * 4 + 1024;   // + alignment slack
};

// One epilogue thread's share of a finished tile: accumulator row `row` (of M live rows),
// columns nt * BN .. nt * BN + BN - 1, read from TMEM at taddr once acc_full completes its
// phase `parity`. Returns false when that wait runs out.
template <int BN, int EPI>
__device__ __forceinline__ bool gemm_epilogue(const GemmParams& p, int M, int row, int nt,
                                              uint32_t taddr, uint64_t* acc_full,
                                              uint32_t parity, float* sgate) {
  const bool row_ok = row < M;
  if constexpr (EPI == EPI_RESID) {
    // the tile's gate slice, the same for every row, staged by each epilogue warp in its own
    // copy in shared memory while the MMAs run, so no chunk of the epilogue waits on a
    // global load (a copy per warp: no barrier across warps, whose bounded waits may end
    // differently)
    const int lane = threadIdx.x & 31;
    sgate += ((threadIdx.x >> 5) & 3) * BN;
    __syncwarp();
    for (int i = lane; i < BN; i += 32) sgate[i] = nt * BN + i < p.N ? p.gate[nt * BN + i] : 0.f;
    __syncwarp();
    // The residual slice of this thread's row is loaded while the MMAs run, so the
    // epilogue waits on no global load once the accumulator is ready.
    const int out_row = !row_ok ? -1 : (p.row_pos != nullptr ? p.row_pos[row] : row);
    const bool live = out_row >= 0;
    uint4 hreg[BN / 8];
    const uint4* h4 = reinterpret_cast<const uint4*>(p.h + (size_t)row * p.N + nt * BN);
#pragma unroll
    for (int j = 0; j < BN / 8; ++j)
      hreg[j] = (live && nt * BN + 8 * j < p.N) ? h4[j] : make_uint4(0, 0, 0, 0);
    // each lane octet stores its eight rows through a transpose, one row's 128 bytes a store
    int orow[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) orow[j] = __shfl_sync(0xffffffffu, out_row, (lane & ~7) + j);
    uint16_t* dst = p.row_pos != nullptr ? p.h_out : p.h;
    if (!mbar_wait(acc_full, parity, ERR_WAIT_MMA)) return false;
    tc_fence_after();
    const float4* g4 = reinterpret_cast<const float4*>(sgate);
#pragma unroll
    for (int c = 0; c < BN / 64; ++c) {
      float v[64];
      tmem_ld32(taddr + c * 64, *reinterpret_cast<float (*)[32]>(&v[0]));
      tmem_ld32(taddr + c * 64 + 32, *reinterpret_cast<float (*)[32]>(&v[32]));
      tmem_ld_wait();
      uint4 w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 hv = hreg[8 * c + j];
        const float4 ga = g4[16 * c + 2 * j];
        const float4 gb = g4[16 * c + 2 * j + 1];
        w[j].x = pack_bf16x2(bf16lo_to_f32(hv.x) + ga.x * v[8 * j + 0],
                             bf16hi_to_f32(hv.x) + ga.y * v[8 * j + 1]);
        w[j].y = pack_bf16x2(bf16lo_to_f32(hv.y) + ga.z * v[8 * j + 2],
                             bf16hi_to_f32(hv.y) + ga.w * v[8 * j + 3]);
        w[j].z = pack_bf16x2(bf16lo_to_f32(hv.z) + gb.x * v[8 * j + 4],
                             bf16hi_to_f32(hv.z) + gb.y * v[8 * j + 5]);
        w[j].w = pack_bf16x2(bf16lo_to_f32(hv.w) + gb.z * v[8 * j + 6],
                             bf16hi_to_f32(hv.w) + gb.w * v[8 * j + 7]);
      }
      octet_transpose(w, lane & 7);
      const int col = nt * BN + 64 * c + 8 * (lane & 7);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (orow[j] >= 0 && col + 8 <= p.N)
          *reinterpret_cast<uint4*>(dst + (size_t)orow[j] * p.N + col) = w[j];
    }
    return true;
  }
  if constexpr (EPI == EPI_QKV) {
    // 64-column chunks (q, k and v each start on a multiple of 64 columns), stored through
    // the octet transpose like the residual epilogue
    const int lane = threadIdx.x & 31;
    if (!mbar_wait(acc_full, parity, ERR_WAIT_MMA)) return false;
    tc_fence_after();
    const int rb = row - (lane & 7);   // the octet's first row
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      float v[64];
      tmem_ld32(taddr + c * 64, *reinterpret_cast<float (*)[32]>(&v[0]));
      tmem_ld32(taddr + c * 64 + 32, *reinterpret_cast<float (*)[32]>(&v[32]));
      tmem_ld_wait();
      uint4 w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        w[j] = make_uint4(pack_bf16x2(v[8 * j + 0], v[8 * j + 1]),
                          pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                          pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                          pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
      octet_transpose(w, lane & 7);
      const int col0 = nt * BN + 64 * c;
      if (col0 >= p.N) continue;
      uint16_t* base;
      int width, cl;
      if (col0 < p.nq) {
        base = p.q; width = p.nq; cl = col0;
      } else if (col0 < p.nq + p.nk) {
        base = p.k; width = p.nk; cl = col0 - p.nq;
      } else {
        base = p.v; width = p.nk; cl = col0 - p.nq - p.nk;
      }
      cl += 8 * (lane & 7);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (rb + j < M)
          *reinterpret_cast<uint4*>(base + (size_t)(rb + j) * width + cl) = w[j];
    }
    return true;
  }
  if (!mbar_wait(acc_full, parity, ERR_WAIT_MMA)) return false;
  tc_fence_after();

  float run_max = -INFINITY, run_sum = 0.f;
  int run_arg = 0;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tmem_ld32(taddr + c * 32, v);
    tmem_ld_wait();
    const int col0 = nt * BN + c * 32;
    if constexpr (EPI == EPI_LMHEAD) {
      // chunk maximum (lowest column on ties), then exp-sum relative to the running max
      float cmax = -INFINITY;
      int carg = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (col0 + j >= p.N) v[j] = -INFINITY;
        if (v[j] > cmax) {
          cmax = v[j];
          carg = j;
        }
      }
      if (cmax > run_max) {
        if (run_max != -INFINITY) run_sum *= ex2_approx((run_max - cmax) * 1.4426950408889634f);
        run_max = cmax;
        run_arg = col0 + carg;
      }
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) s += ex2_approx((v[j] - run_max) * 1.4426950408889634f);
      run_sum += s;
    } else if constexpr (EPI == EPI_QKV_ROPE) {
      if (row_ok && col0 < p.N && col0 < p.nq + p.nk) {
        // the 32 columns of a chunk lie in one head (head_dim is 64 or 128)
        const int hd0 = (col0 < p.nq ? col0 : col0 - p.nq) % p.head_dim;
        const float2* cs = p.rope_cs + (size_t)row * (p.head_dim / 2) + hd0 / 2;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 c = __ldg(&cs[j]);
          const float a = v[2 * j], b = v[2 * j + 1];
          v[2 * j] = a * c.x - b * c.y;
          v[2 * j + 1] = a * c.y + b * c.x;
        }
      }
      if (row_ok && col0 < p.N) {
        uint16_t* dst;
        if (col0 < p.nq)
          dst = p.q + (size_t)row * p.nq + col0;
        else if (col0 < p.nq + p.nk)
          dst = p.k + (size_t)row * p.nk + (col0 - p.nq);
        else
          dst = p.v + (size_t)row * p.nk + (col0 - p.nq - p.nk);
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 w;
          w.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
          w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
          w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
          w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
          d4[j] = w;
        }
      }
    }
  }
  if constexpr (EPI == EPI_LMHEAD) {
    if (row_ok) {
      const size_t o = (size_t)row * p.n_tiles + nt;
      p.part_max[o] = run_max;
      p.part_arg[o] = run_arg;
      p.part_sum[o] = run_sum;
    }
  }
  return true;
}

template <int BN, int STAGES, int EPI>
__global__ void __launch_bounds__(256, 1)
    gemm_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
  using L = GemmSmem<BN, STAGES>;
  if (p.skip != nullptr && *p.skip != 0) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkb = p.K / 64;
  const int M = p.m_count != nullptr ? min(max(*p.m_count, 0), p.M) : p.M;
  const int m_tiles = (M + 127) / 128;
  const int items = m_tiles * p.n_tiles;
  if (blockIdx.x >= items) return;   // before any barrier or TMEM allocation

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 128);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
        const int mt = item % m_tiles;
        const int nt = item / m_tiles;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (it >= STAGES && !mbar_wait(&empty[s], ph ^ 1, ERR_WAIT_MMA)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * L::kStageBytes;
          mbar_arrive_expect_tx(&full[s], L::kStageBytes);
          tma_load_2d(sa, &tmA, &full[s], kb * 64, mt * 128);
          tma_load_2d(sa + L::kABytes, &tmB, &full[s], kb * 64, nt * BN);
        }
      }
      // On an aborted run, wait (bounded) for the loads still in flight before leaving.
      if (!ok) {
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          mbar_wait_drain(&full[j % STAGES], (j / STAGES) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, BN, 0);
      int it = 0, lt = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < items && ok; item += gridDim.x, ++lt) {
        const int acc = lt & 1;
        const int use = lt >> 1;
        if (lt >= 2 && !mbar_wait(&acc_empty[acc], (use & 1) ^ 1, ERR_WAIT_EPI)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&full[s], (it / STAGES) & 1, ERR_WAIT_TMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * L::kStageBytes);
          const uint32_t b0 = a0 + L::kABytes;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            mma_bf16_ss(d_tmem, sdesc_sw128(a0 + k * 32, 16, 1024),
                        sdesc_sw128(b0 + k * 32, 16, 1024), idesc, (kb | k) != 0);
          }
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&acc_full[acc]);
      }
      // Let every MMA issued so far finish before the TMEM is released.
      if (it > 0) mbar_wait_drain(&empty[(it - 1) % STAGES], ((it - 1) / STAGES) & 1);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    int lt = 0;
    for (int item = blockIdx.x; item < items; item += gridDim.x, ++lt) {
      const int mt = item % m_tiles;
      const int nt = item / m_tiles;
      const int acc = lt & 1;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      if (!gemm_epilogue<BN, EPI>(p, M, mt * 128 + q * 32 + lane, nt, taddr, &acc_full[acc],
                                  (lt >> 1) & 1,
                                  reinterpret_cast<float*>(smem + L::kGateOffset)))
        break;
      tc_fence_before();
      mbar_arrive(&acc_empty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * BN);
  }
}

// ------------------------------------------------------------------------------------------
// Pair variant: a cluster of two CTAs on the two SMs of a TPC computes 256 x 256 tiles with
// tcgen05.mma.cta_group::2 (M = 256), issued by the even CTA. Each CTA stages its own 128
// rows of A and its own 128 rows of B (half of the tile's N) per 64-wide k step, so an SM
// takes in 32 KB per k step instead of the 48 KB of a single-CTA 128 x 256 tile for the same
// tensor work per SM; each CTA's TMEM receives its 128 rows of the 256-column accumulator
// and its epilogue warps run the same epilogue as above. Both CTAs' TMA bytes complete on
// the even CTA's `full` barriers; MMA completions are multicast to both CTAs' `empty` and
// `acc_full` barriers; the epilogue warps of both CTAs arrive (one arrive per warp) on the
// even CTA's `acc_empty`.
// ------------------------------------------------------------------------------------------
// Ring depth: seven 32 KB stages where the shared memory allows, six for the residual
// epilogue, which also keeps the gate slices there.
__host__ __device__ constexpr int pair_gemm_stages(int epi) { return epi == EPI_RESID ? 6 : 7; }

template <int STAGES, int EPI>
struct GemmPairSmem {
  static constexpr int kABytes = 128 * 128;      // this CTA's 128 rows of A x 64 bf16
  static constexpr int kBBytes = 128 * 128;      // this CTA's 128 rows of B x 64 bf16
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOffset = STAGES * kStageBytes;
  static constexpr int kGateOffset = kBarOffset + 256;     // gate slices (EPI_RESID), 4 warps
  static constexpr int kBytes = kGateOffset + (EPI == EPI_RESID ? 4 * 256 * 4 : 0) + 1024;
};

template <int STAGES, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  using L = GemmPairSmem<STAGES, EPI>;
  constexpr int BN = 256;
  if (p.skip != nullptr && *p.skip != 0) return;   // both CTAs of a pair read the same flag
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);   // even CTA's used
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;                                    // even CTA's used
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkb = p.K / 64;
  const int M = p.m_count != nullptr ? min(max(*p.m_count, 0), p.M) : p.M;
  const int m_pairs = (M + 255) / 256;
  const int items = m_pairs * p.n_tiles;
  const int cluster = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;
  if (cluster >= items) return;   // both CTAs alike, before any barrier or TMEM allocation

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 8);   // 4 epilogue warps x 2 CTAs
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 2 * BN);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before any cross-CTA arrival or byte count
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producers
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int item = cluster; item < items && ok; item += n_clusters) {
        const int mp = item % m_pairs;
        const int nt = item / m_pairs;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (it >= STAGES && !mbar_wait(&empty[s], ph ^ 1, ERR_WAIT_MMA)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * L::kStageBytes;
          const uint32_t bar = cluster_addr(&full[s], 0);
          if (even) mbar_arrive_expect_tx(&full[s], 2 * L::kStageBytes);   // both CTAs
          tma_load_2d_pair(sa, &tmA, bar, kb * 64, mp * 256 + (int)rank * 128);
          tma_load_2d_pair(sa + L::kABytes, &tmB, bar, kb * 64, nt * BN + (int)rank * 128);
        }
      }
      // On an aborted run, wait (bounded) for the loads still in flight before leaving.
      if (!ok && even) {
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          mbar_wait_drain(&full[j % STAGES], (j / STAGES) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (even)
    if (even && lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(256, BN, 0);
      int it = 0, lt = 0;
      bool ok = true;
      for (int item = cluster; item < items && ok; item += n_clusters, ++lt) {
        const int acc = lt & 1;
        const int use = lt >> 1;
        if (lt >= 2 && !mbar_wait(&acc_empty[acc], (use & 1) ^ 1, ERR_WAIT_EPI)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&full[s], (it / STAGES) & 1, ERR_WAIT_TMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * L::kStageBytes);
          const uint32_t b0 = a0 + L::kABytes;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            mma_pair_ss(d_tmem, sdesc_sw128(a0 + k * 32, 16, 1024),
                        sdesc_sw128(b0 + k * 32, 16, 1024), idesc, (kb | k) != 0);
          }
          mma_commit_pair(&empty[s], 0x3);
        }
        if (!ok) break;
        mma_commit_pair(&acc_full[acc], 0x3);
      }
      // Let every MMA issued so far finish before the TMEM is released.
      if (it > 0) mbar_wait_drain(&empty[(it - 1) % STAGES], ((it - 1) / STAGES) & 1);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue (both)
    const int q = warp & 3;
    int lt = 0;
    for (int item = cluster; item < items; item += n_clusters, ++lt) {
      const int mp = item % m_pairs;
      const int nt = item / m_pairs;
      const int acc = lt & 1;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      if (!gemm_epilogue<BN, EPI>(p, M, mp * 256 + (int)rank * 128 + q * 32 + lane, nt, taddr,
                                  &acc_full[acc], (lt >> 1) & 1,
                                  reinterpret_cast<float*>(smem + L::kGateOffset)))
        break;
      // the accumulator is free once all four warps of both CTAs have read it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (even) mbar_arrive(&acc_empty[acc]);
        else mbar_arrive_cluster_relaxed(cluster_addr(&acc_empty[acc], 0));
      }
    }
  }

  // No CTA of the pair leaves (or frees its TMEM) while the other may still signal its
  // barriers or while pair MMAs may still write its TMEM.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 2 * BN);
  }
}

}  // namespace td
