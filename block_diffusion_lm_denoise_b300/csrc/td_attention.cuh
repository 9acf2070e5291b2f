// td_attention.cuh -- fused block attention of the denoiser
// ("NVIDIA、Nemotron-Labs-TwoTowerを公開…", news.chathome.org, inference paragraph: the block
// attends bidirectionally to itself and, layer by layer, to the context tower's KV cache).
//
// One CTA row group = the S block tokens x Gc query heads that share one KV head (GQA), i.e.
// R = S*Gc <= 256 query rows; they are two 128-row MMA halves that read every K/V byte once.
// Keys are visited in 64-key tiles: ceil(Lmax/64) context tiles, then one tile holding the
// S block keys; one online softmax runs over all of them (one joint softmax per row).
// The (row group, tile) space is flattened and cut into gridDim.x equal contiguous ranges
// (split-K over the context, balanced across the SMs); a CTA whose range covers a whole row
// group writes the normalised bf16 output directly, otherwise it writes an unnormalised
// partial (O, running max, running sum) that attn_merge_kernel combines by log-sum-exp.
//
// Roles (320 threads): warps 0-3 = softmax/epilogue of rows 0-127, warps 4-7 = rows 128-255,
// warp 8 lane 0 = TMA producer, warp 9 = TMEM allocator + (lane 0) MMA issuer.
// TMEM (512 columns): O[h] at columns 128h (fp32, D columns), S[h][buf] at 256 + 64(2h+buf).
// Per tile: S[h] = Q[h] K^T (M=128, N=64, K=D), softmax warps turn S into bf16 P in shared
// memory (128-byte swizzled K-major rows), then O[h] += P V (M=128, N=D, K=64, V read
// MN-major straight from the TMA tile). The MMA of S for tile n+1 is issued before the PV
// MMA of tile n, so the tensor pipe works while the softmax warps compute exponentials.
// Rescaling of O is lazy: the running max only moves when a tile's max exceeds it by more
// than 8 (log2 units), so P stays <= 2^8 and the TMEM round trip is rare.
#pragma once

#include "td_ptx.cuh"

namespace td {

struct AttnParams {
  int B, S, Hq, Hkv, D, Lmax;
  int G, Gc, NC, R;          // heads per KV head, heads per row group, row groups per KV head
  int n_ctx_tiles, T;        // ceil(Lmax/64), T = n_ctx_tiles + 1
  int n_groups;              // B * Hkv * NC
  long long total;           // n_groups * T
  int max_seg;               // partial-record slots per CTA
  const int* ctx_len;        // [B] or null
  float* part_o;             // [gridDim.x * max_seg][R][D]
  float* part_ml;            // [gridDim.x * max_seg][R][2]  (max in log2 units, sum)
  uint16_t* out;             // [B, S, Hq, D] bf16
  float* lse;                // [B, S, Hq] or null
  float scale_log2;          // log2(e) / sqrt(D)
};

constexpr int kAttnStages = 3;
constexpr int kAttnThreads = 320;

template <int D>
struct AttnSmem {
  static constexpr int kQRegion = 256 * 128;                  // 256 rows x 64 bf16, per d-half
  static constexpr int kQBytes = kQRegion * (D / 64);
  static constexpr int kKVHalf = 64 * 128;                    // 64 keys x 64 bf16
  static constexpr int kKBytes = kKVHalf * (D / 64);
  static constexpr int kStageBytes = 2 * kKBytes;             // K then V
  static constexpr int kPBytes = 128 * 128;                   // 128 rows x 64 bf16, per half
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQBytes;
  static constexpr int kOffP = kOffKV + kAttnStages * kStageBytes;
  static constexpr int kOffBar = kOffP + 2 * kPBytes;
  static constexpr int kBytes = kOffBar + 512 + 1024;
};

__device__ __forceinline__ long long attn_lo(long long c, long long total, int ncta) {
  return c * total / ncta;
}

// Per-CTA iteration over row-group segments and the tiles that carry work.
struct SegInfo {
  int grp;        // row-group index
  int b, g, chunk;
  int t0, t1;     // tile range [t0, t1) of this segment within the row group
  int L;          // valid context length of sequence b
  int nvt;        // context tiles holding valid keys: ceil(L / 64)
  bool full;      // the segment covers the whole row group
};

__device__ __forceinline__ SegInfo attn_seg(const AttnParams& p, long long lo, long long hi,
                                            int grp) {
  SegInfo s;
  s.grp = grp;
  const int per_b = p.Hkv * p.NC;
  s.b = grp / per_b;
  s.g = (grp % per_b) / p.NC;
  s.chunk = grp % p.NC;
  const long long base = (long long)grp * p.T;
  s.t0 = (int)((lo > base ? lo : base) - base);
  s.t1 = (int)((hi < base + p.T ? hi : base + p.T) - base);
  s.L = p.ctx_len ? min(max(p.ctx_len[s.b], 0), p.Lmax) : p.Lmax;
  s.nvt = (s.L + 63) / 64;
  s.full = (s.t0 == 0 && s.t1 == p.T);
  return s;
}

// The t-th tile of a row group carries work if it is a context tile with valid keys or the
// block tile (t == n_ctx_tiles).
__device__ __forceinline__ bool attn_tile_live(const AttnParams& p, const SegInfo& s, int t) {
  return (t < p.n_ctx_tiles) ? (t < s.nvt) : true;
}

__device__ __forceinline__ int attn_seg_work(const AttnParams& p, const SegInfo& s) {
  int n = 0;
  const int ctx_end = s.t1 < s.nvt ? s.t1 : s.nvt;
  if (ctx_end > s.t0) n += ctx_end - (s.t0 < p.n_ctx_tiles ? s.t0 : p.n_ctx_tiles);
  if (s.t0 <= p.n_ctx_tiles && p.n_ctx_tiles < s.t1) n += 1;
  return n;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fused_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmKc,
                      const __grid_constant__ CUtensorMap tmVc,
                      const __grid_constant__ CUtensorMap tmKb,
                      const __grid_constant__ CUtensorMap tmVb, const AttnParams p) {
  using L = AttnSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sKV = smem + L::kOffKV;
  uint8_t* sP = smem + L::kOffP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* kv_full = bars;                       // [3]
  uint64_t* kv_empty = bars + 3;                  // [3]
  uint64_t* q_full = bars + 6;
  uint64_t* q_empty = bars + 7;
  uint64_t* s_full = bars + 8;                    // [h*2 + buf]
  uint64_t* s_empty = bars + 12;                  // [h*2 + buf]
  uint64_t* p_full = bars + 16;                   // [h]
  uint64_t* o_done = bars + 18;                   // [h]
  uint64_t* o_free = bars + 20;                   // [h]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 24);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NH = (p.R + 127) / 128;   // 1 or 2 MMA halves
  const long long lo = attn_lo(blockIdx.x, p.total, gridDim.x);
  const long long hi = attn_lo(blockIdx.x + 1, p.total, gridDim.x);
  const int grp_first = (int)(lo / p.T);
  const int grp_last = (int)((hi - 1) / p.T);

  // Zero the tiles once: rows that no TMA box covers (padding query rows, block-key rows
  // beyond S) must hold finite values because P = 0 multiplies them.
  {
    uint4* z = reinterpret_cast<uint4*>(smem);
    const int n16 = L::kOffBar / 16;
    for (int i = threadIdx.x; i < n16; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kAttnStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 128);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&p_full[h], 128);
      mbar_init(&o_done[h], 1);
      mbar_init(&o_free[h], 128);
    }
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmKc);
      tma_prefetch_desc(&tmVc);
      tma_prefetch_desc(&tmKb);
      tma_prefetch_desc(&tmVb);
      int n = 0, sgw = 0;
      bool ok = true;
      for (int grp = grp_first; grp <= grp_last && ok; ++grp) {
        const SegInfo s = attn_seg(p, lo, hi, grp);
        if (attn_seg_work(p, s) == 0) continue;
        if (sgw >= 1 && !mbar_wait(q_empty, (sgw - 1) & 1, ERR_WAIT_MMA)) { ok = false; break; }
        mbar_arrive_expect_tx(q_full, p.R * 128 * (D / 64));
        for (int kh = 0; kh < D / 64; ++kh)
          tma_load_4d(sQ + kh * L::kQRegion, &tmQ, q_full, kh * 64, s.g * p.G + s.chunk * p.Gc,
                      0, s.b);
        ++sgw;
        for (int t = s.t0; t < s.t1; ++t) {
          if (!attn_tile_live(p, s, t)) continue;
          const int st = n % kAttnStages;
          if (n >= kAttnStages &&
              !mbar_wait(&kv_empty[st], ((n / kAttnStages) & 1) ^ 1, ERR_WAIT_MMA)) {
            ok = false;
            break;
          }
          uint8_t* sk = sKV + st * L::kStageBytes;
          uint8_t* sv = sk + L::kKBytes;
          if (t < p.n_ctx_tiles) {
            mbar_arrive_expect_tx(&kv_full[st], 2 * 64 * 128 * (D / 64));
            const int row3 = s.b * p.Hkv + s.g;
            for (int kh = 0; kh < D / 64; ++kh) {
              tma_load_3d(sk + kh * L::kKVHalf, &tmKc, &kv_full[st], kh * 64, t * 64, row3);
              tma_load_3d(sv + kh * L::kKVHalf, &tmVc, &kv_full[st], kh * 64, t * 64, row3);
            }
          } else {
            mbar_arrive_expect_tx(&kv_full[st], 2 * p.S * 128 * (D / 64));
            for (int kh = 0; kh < D / 64; ++kh) {
              tma_load_4d(sk + kh * L::kKVHalf, &tmKb, &kv_full[st], kh * 64, s.g, 0, s.b);
              tma_load_4d(sv + kh * L::kKVHalf, &tmVb, &kv_full[st], kh * 64, s.g, 0, s.b);
            }
          }
          ++n;
        }
      }
      if (!ok) {
        for (int j = (n > kAttnStages ? n - kAttnStages : 0); j < n; ++j)
          mbar_wait(&kv_full[j % kAttnStages], (j / kAttnStages) & 1, ERR_WAIT_TMA);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, 64, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, 1);
      bool ok = true;
      int n = 0, sgw = 0, issued = 0;
      // pending PV: the previous work tile
      int pv_n = -1, pv_st = 0, pv_first = 0, pv_sgw = 0;
      auto issue_pv = [&](int m, int st, int first, int sg) -> bool {
        for (int h = 0; h < NH; ++h) {
          if (!mbar_wait(&p_full[h], m & 1, ERR_WAIT_EPI)) return false;
          if (first && sg >= 1 && !mbar_wait(&o_free[h], (sg - 1) & 1, ERR_WAIT_EPI)) return false;
          tc_fence_after();
          const uint32_t pa = smem_u32(sP + h * L::kPBytes);
          const uint32_t vb = smem_u32(sKV + st * L::kStageBytes + L::kKBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            mma_bf16_ss(tmem + h * 128, sdesc_sw128(pa + kk * 32, 16, 1024),
                        sdesc_sw128(vb + kk * 2048, L::kKVHalf, 1024), idesc_pv,
                        !(first && kk == 0));
          }
          mma_commit(&o_done[h]);
        }
        mma_commit(&kv_empty[st]);
        ++issued;
        return true;
      };
      for (int grp = grp_first; grp <= grp_last && ok; ++grp) {
        const SegInfo s = attn_seg(p, lo, hi, grp);
        const int nwork = attn_seg_work(p, s);
        if (nwork == 0) continue;
        int wi = 0;
        for (int t = s.t0; t < s.t1 && ok; ++t) {
          if (!attn_tile_live(p, s, t)) continue;
          const int st = n % kAttnStages;
          const int first = (wi == 0), last = (wi == nwork - 1);
          if (!mbar_wait(&kv_full[st], (n / kAttnStages) & 1, ERR_WAIT_TMA)) { ok = false; break; }
          if (first && !mbar_wait(q_full, sgw & 1, ERR_WAIT_TMA)) { ok = false; break; }
          tc_fence_after();
          const int buf = n & 1;
          for (int h = 0; h < NH; ++h) {
            if (n >= 2 &&
                !mbar_wait(&s_empty[h * 2 + buf], ((n >> 1) - 1) & 1, ERR_WAIT_EPI)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sacc = tmem + 256 + (h * 2 + buf) * 64;
            const uint32_t qa = smem_u32(sQ + h * 128 * 128);
            const uint32_t kb = smem_u32(sKV + st * L::kStageBytes);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int kh = kk >> 2, k4 = kk & 3;
              mma_bf16_ss(sacc, sdesc_sw128(qa + kh * L::kQRegion + k4 * 32, 16, 1024),
                          sdesc_sw128(kb + kh * L::kKVHalf + k4 * 32, 16, 1024), idesc_qk,
                          kk != 0);
            }
            mma_commit(&s_full[h * 2 + buf]);
          }
          if (!ok) break;
          if (last) mma_commit(q_empty);
          if (pv_n >= 0 && !issue_pv(pv_n, pv_st, pv_first, pv_sgw)) { ok = false; break; }
          pv_n = n; pv_st = st; pv_first = first; pv_sgw = sgw;
          ++n;
          ++wi;
        }
        ++sgw;
      }
      if (ok && pv_n >= 0) ok = issue_pv(pv_n, pv_st, pv_first, pv_sgw);
      // Let every MMA issued so far finish before the TMEM is released.
      if (n > 0) {
        const int j = n - 1;
        mbar_wait(&s_full[(0 * 2) + (j & 1)], (j >> 1) & 1, ERR_WAIT_MMA);
      }
      if (issued > 0) {
        const int j = issued - 1;
        for (int h = 0; h < NH; ++h) mbar_wait(&o_done[h], j & 1, ERR_WAIT_MMA);
      }
    }
    __syncwarp();
  } else {
    // ================================================================ softmax / epilogue
    const int h = warp >> 2;              // MMA half
    const int q4 = warp & 3;              // TMEM lane quarter
    const int r = h * 128 + q4 * 32 + lane;
    const bool row_ok = r < p.R;
    const bool half_live = h < NH;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float sc = p.scale_log2;
    int n = 0;
    bool ok = true;
    float m_run = -INFINITY, l_run = 0.f;
    for (int grp = grp_first; grp <= grp_last && ok; ++grp) {
      const SegInfo s = attn_seg(p, lo, hi, grp);
      const int nwork = attn_seg_work(p, s);
      const int s_tok = r / p.Gc;
      const int head = s.g * p.G + s.chunk * p.Gc + (r % p.Gc);
      const int rec = blockIdx.x * p.max_seg + (grp - grp_first);
      if (nwork == 0 || !half_live) {
        // No key reaches this segment (or this half has no rows): an empty partial.
        if (half_live && row_ok && !s.full) {
          p.part_ml[((size_t)rec * p.R + r) * 2 + 0] = -INFINITY;
          p.part_ml[((size_t)rec * p.R + r) * 2 + 1] = 0.f;
        }
        if (nwork != 0) n += nwork;
        continue;
      }
      int wi = 0;
      for (int t = s.t0; t < s.t1 && ok; ++t) {
        if (!attn_tile_live(p, s, t)) continue;
        const int first = (wi == 0), last = (wi == nwork - 1);
        const int buf = n & 1;
        if (!mbar_wait(&s_full[h * 2 + buf], (n >> 1) & 1, ERR_WAIT_MMA)) { ok = false; break; }
        tc_fence_after();
        float x[64];
        {
          float a[32], b2[32];
          const uint32_t sacc = tmem + lane_off + 256 + (h * 2 + buf) * 64;
          tmem_ld32(sacc, a);
          tmem_ld32(sacc + 32, b2);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) { x[j] = a[j]; x[32 + j] = b2[j]; }
        }
        tc_fence_before();
        mbar_arrive(&s_empty[h * 2 + buf]);
        const int nvalid = (t < p.n_ctx_tiles) ? min(64, s.L - t * 64) : p.S;
        float tmax = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          x[j] = (j < nvalid) ? x[j] * sc : -INFINITY;
          tmax = fmaxf(tmax, x[j]);
        }
        bool waited = false;
        if (first) {
          m_run = tmax;
          l_run = 0.f;
        } else if (tmax > m_run + 8.0f) {
          const float alpha = ex2_approx(m_run - tmax);
          m_run = tmax;
          l_run *= alpha;
          if (!mbar_wait(&o_done[h], (n - 1) & 1, ERR_WAIT_MMA)) { ok = false; break; }
          waited = true;
          tc_fence_after();
          const uint32_t oacc = tmem + lane_off + h * 128;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(oacc + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] *= alpha;
            tmem_st32(oacc + c * 32, o);
          }
          tmem_st_wait();
        }
        // P = 2^(x - m) rounded to bf16; the row sum adds the rounded values
        uint32_t pk[32];
        float lsum = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float e0 = ex2_approx(x[2 * j] - m_run);
          const float e1 = ex2_approx(x[2 * j + 1] - m_run);
          pk[j] = pack_bf16x2(e0, e1);
          lsum += bf16lo_to_f32(pk[j]) + bf16hi_to_f32(pk[j]);
        }
        l_run += lsum;
        if (n >= 1 && !waited && !mbar_wait(&o_done[h], (n - 1) & 1, ERR_WAIT_MMA)) {
          ok = false;
          break;
        }
        {
          // row r of this half: 128 bytes, eight 16-byte chunks XOR-swizzled by (row & 7)
          const int rr = q4 * 32 + lane;
          uint8_t* prow = sP + h * L::kPBytes + rr * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 w = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            *reinterpret_cast<uint4*>(prow + ((c ^ (rr & 7)) << 4)) = w;
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[h]);
        if (last) {
          if (!mbar_wait(&o_done[h], n & 1, ERR_WAIT_MMA)) { ok = false; break; }
          tc_fence_after();
          const uint32_t oacc = tmem + lane_off + h * 128;
          if (s.full) {
            const float inv = 1.f / l_run;
            uint16_t* dst = p.out + (((size_t)s.b * p.S + s_tok) * p.Hq + head) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              float o[32];
              tmem_ld32(oacc + c * 32, o);
              tmem_ld_wait();
              if (row_ok) {
                uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  d4[j] = make_uint4(pack_bf16x2(o[8 * j] * inv, o[8 * j + 1] * inv),
                                     pack_bf16x2(o[8 * j + 2] * inv, o[8 * j + 3] * inv),
                                     pack_bf16x2(o[8 * j + 4] * inv, o[8 * j + 5] * inv),
                                     pack_bf16x2(o[8 * j + 6] * inv, o[8 * j + 7] * inv));
              }
            }
            if (row_ok && p.lse)
              p.lse[((size_t)s.b * p.S + s_tok) * p.Hq + head] =
                  (m_run + __log2f(l_run)) * 0.6931471805599453f;
          } else {
            float* dst = p.part_o + ((size_t)rec * p.R + r) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              float o[32];
              tmem_ld32(oacc + c * 32, o);
              tmem_ld_wait();
              if (row_ok) {
                float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  d4[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
              }
            }
            if (row_ok) {
              p.part_ml[((size_t)rec * p.R + r) * 2 + 0] = m_run;
              p.part_ml[((size_t)rec * p.R + r) * 2 + 1] = l_run;
            }
          }
          tc_fence_before();
          mbar_arrive(&o_free[h]);
        }
        ++n;
        ++wi;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Log-sum-exp merge of the partials of every row group that no single CTA covered.
// One CTA per row group; thread (row, 4 columns).
__global__ void attn_merge_kernel(const AttnParams p, int ncta) {
  const int grp = blockIdx.x;
  const long long first_tile = (long long)grp * p.T;
  const long long last_tile = first_tile + p.T - 1;
  // CTA owning a tile x: the largest c with lo(c) <= x (lo is monotone in c)
  auto owner = [&](long long x) {
    int a = 0, b = ncta - 1;
    while (a < b) {
      const int mid = (a + b + 1) >> 1;
      if (attn_lo(mid, p.total, ncta) <= x) a = mid; else b = mid - 1;
    }
    return a;
  };
  const int c0 = owner(first_tile);
  const int c1 = owner(last_tile);
  if (c0 == c1) return;   // written directly by its only CTA
  const int per_b = p.Hkv * p.NC;
  const int b = grp / per_b;
  const int g = (grp % per_b) / p.NC;
  const int chunk = grp % p.NC;
  const int D = p.D;
  const int nq4 = D / 4;
  for (int idx = threadIdx.x; idx < p.R * nq4; idx += blockDim.x) {
    const int r = idx / nq4;
    const int d4 = idx % nq4;
    float M = -INFINITY;
    for (int c = c0; c <= c1; ++c) {
      const int rec = c * p.max_seg + (grp - (int)(attn_lo(c, p.total, ncta) / p.T));
      M = fmaxf(M, p.part_ml[((size_t)rec * p.R + r) * 2]);
    }
    float Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = c0; c <= c1; ++c) {
      const int rec = c * p.max_seg + (grp - (int)(attn_lo(c, p.total, ncta) / p.T));
      const float mk = p.part_ml[((size_t)rec * p.R + r) * 2];
      const float lk = p.part_ml[((size_t)rec * p.R + r) * 2 + 1];
      if (lk == 0.f) continue;
      const float w = exp2f(mk - M);
      Lsum += lk * w;
      const float4 o = reinterpret_cast<const float4*>(p.part_o + ((size_t)rec * p.R + r) * D)[d4];
      acc.x += o.x * w; acc.y += o.y * w; acc.z += o.z * w; acc.w += o.w * w;
    }
    const float inv = 1.f / Lsum;
    const int s_tok = r / p.Gc;
    const int head = g * p.G + chunk * p.Gc + (r % p.Gc);
    uint16_t* dst = p.out + (((size_t)b * p.S + s_tok) * p.Hq + head) * D + d4 * 4;
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    if (d4 == 0 && p.lse)
      p.lse[((size_t)b * p.S + s_tok) * p.Hq + head] = (M + log2f(Lsum)) * 0.6931471805599453f;
  }
}

}  // namespace td
