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
// Roles (608 threads): warps 0-7 = softmax/epilogue of rows 0-127 (two warps per 32 rows,
// one per half of each 64-key tile), warps 8-15 = rows 128-255, warp 16 lane 0 = TMA
// producer, warps 17-20 lane 0 = MMA issuers: S = Q K^T of rows 0-127 / 128-255 (17, 18)
// and O += P V of rows 0-127 / 128-255 (19, 20); warp 17 also owns the TMEM allocation.
// A tcgen05.mma issue costs about a hundred cycles and a tile needs twelve per half, so the
// issue is spread over four threads; the four streams touch disjoint TMEM columns.
// TMEM (512 columns): O[h] at columns 128h (fp32, D columns); S[h] at 256 + 64h (fp32, 64
// keys); P[h][buf] at 384 + 32(2h+buf) (bf16 probabilities, two per column).
// Per tile n: S[h] = Q[h] K^T (M=128, N=64, K=D); the softmax warps read S and write P into
// buffer n&1; O[h] += P V is issued with A = P from TMEM and B = V read MN-major straight
// from the TMA tile. As soon as the softmax warps have read S(n) the MMA warp issues S for
// tile n+1, which runs on the tensor pipe while they compute exponentials, and P is double
// buffered, so the softmax warps never wait on the PV of the previous tile.
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

constexpr int kAttnStages = 4;
constexpr int kAttnThreads = 672;   // 16 softmax warps + producer + 4 MMA issuers
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;        // first MMA issuer warp; also allocates the TMEM
// warps 17, 18: S = Q K^T for halves 0, 1; warps 19, 20: O += P V for halves 0, 1

template <int D>
struct AttnSmem {
  static constexpr int kQRegion = 256 * 128;                  // 256 rows x 64 bf16, per d-half
  static constexpr int kQBytes = kQRegion * (D / 64);
  static constexpr int kKVHalf = 64 * 128;                    // 64 keys x 64 bf16
  static constexpr int kKBytes = kKVHalf * (D / 64);
  static constexpr int kStageBytes = 2 * kKBytes;             // K then V
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQBytes;
  static constexpr int kOffX = kOffKV + kAttnStages * kStageBytes;   // row max / sum exchange
  static constexpr int kOffBar = kOffX + 8192;
  static constexpr int kBytes = kOffBar + 512 + 1024;
};

__device__ __forceinline__ void pair_sync(int id) {
  asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

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

// Walks the live tiles of one CTA in order: segment (row group) by segment.
struct TileCursor {
  SegInfo s;
  int grp, t, wi, nwork, sgw;   // sgw: index among segments with work
  bool valid;
};

__device__ __forceinline__ void cursor_next_segment(TileCursor& c, const AttnParams& p,
                                                    long long lo, long long hi, int grp_last) {
  for (++c.grp; c.grp <= grp_last; ++c.grp) {
    const SegInfo s = attn_seg(p, lo, hi, c.grp);
    const int nw = attn_seg_work(p, s);
    if (nw > 0) {
      c.s = s;
      c.nwork = nw;
      c.wi = 0;
      ++c.sgw;
      c.t = s.t0;
      while (!attn_tile_live(p, s, c.t)) ++c.t;
      c.valid = true;
      return;
    }
  }
  c.valid = false;
}

__device__ __forceinline__ void cursor_init(TileCursor& c, const AttnParams& p, long long lo,
                                            long long hi, int grp_first, int grp_last) {
  c.grp = grp_first - 1;
  c.sgw = -1;
  c.valid = false;
  cursor_next_segment(c, p, lo, hi, grp_last);
}

__device__ __forceinline__ void cursor_next(TileCursor& c, const AttnParams& p, long long lo,
                                            long long hi, int grp_last) {
  if (c.valid && c.wi + 1 < c.nwork) {
    ++c.t;
    while (!attn_tile_live(p, c.s, c.t)) ++c.t;
    ++c.wi;
    return;
  }
  cursor_next_segment(c, p, lo, hi, grp_last);
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
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* kv_full = bars;                       // [kAttnStages]
  uint64_t* kv_empty = bars + kAttnStages;        // [kAttnStages]
  uint64_t* q_full = bars + 2 * kAttnStages;
  uint64_t* q_empty = q_full + 1;
  uint64_t* s_full = q_full + 2;                  // [h]          S written
  uint64_t* s_empty = s_full + 2;                 // [h]          S read by the softmax warps
  uint64_t* p_full = s_empty + 2;                 // [h*2 + buf]  P written
  uint64_t* o_done = p_full + 4;                  // [h*2 + buf]  PV of a tile using P[buf] done
  uint64_t* o_free = o_done + 4;                  // [h]          O read out at a segment end
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_free + 2);

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
      mbar_init(&kv_empty[i], NH);      // one commit per MMA issuer
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, NH);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&s_full[h], 1);
      mbar_init(&s_empty[h], 256);
      mbar_init(&o_free[h], 256);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&p_full[i], 256);
      mbar_init(&o_done[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
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
  } else if (warp >= kMmaWarp && warp < kMmaWarp + 4) {
    // ================================================================ MMA issuers
    const int role = warp - kMmaWarp;              // 0, 1: QK of half role; 2, 3: PV of half role-2
    const int h = role & 1;
    if (lane == 0 && h < NH) {
      TileCursor c;
      cursor_init(c, p, lo, hi, grp_first, grp_last);
      int n = 0;
      bool ok = true;
      if (role < 2) {
        // ---------------------------------------------------------- S[h] = Q[h] K^T
        constexpr uint32_t idesc_qk = idesc_bf16(128, 64, 0);
        // descriptors of k-step 0; later k-steps add (byte offset >> 4) to the address field
        const uint64_t qdesc = sdesc_sw128(smem_u32(sQ + h * 128 * 128), 16, 1024);
        const uint32_t sacc = tmem + 256 + h * 64;
        for (; c.valid; ++n) {
          const int st = n % kAttnStages;
          if (!mbar_wait(&kv_full[st], (n / kAttnStages) & 1, ERR_WAIT_TMA)) { ok = false; break; }
          if (c.wi == 0 && !mbar_wait(q_full, c.sgw & 1, ERR_WAIT_TMA)) { ok = false; break; }
          if (n >= 1 && !mbar_wait(&s_empty[h], (n - 1) & 1, ERR_WAIT_EPI)) { ok = false; break; }
          tc_fence_after();
          const uint64_t kdesc = sdesc_sw128(smem_u32(sKV + st * L::kStageBytes), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t qa = qdesc + (((kk >> 2) * L::kQRegion + (kk & 3) * 32) >> 4);
            const uint64_t kb = kdesc + (((kk >> 2) * L::kKVHalf + (kk & 3) * 32) >> 4);
            mma_bf16_ss(sacc, qa, kb, idesc_qk, kk != 0);
          }
          mma_commit(&s_full[h]);
          if (c.wi == c.nwork - 1) mma_commit(q_empty);
          cursor_next(c, p, lo, hi, grp_last);
        }
        // Let every MMA issued so far finish before the TMEM is released.
        if (n > 0) mbar_wait(&s_full[h], (n - 1) & 1, ERR_WAIT_MMA);
      } else {
        // ---------------------------------------------------------- O[h] += P[h] V
        constexpr uint32_t idesc_pv = idesc_bf16(128, D, 1);
        for (; c.valid; ++n) {
          const int st = n % kAttnStages;
          const int buf = n & 1;
          const bool first = c.wi == 0;
          if (!mbar_wait(&p_full[h * 2 + buf], (n >> 1) & 1, ERR_WAIT_EPI)) { ok = false; break; }
          if (first && c.sgw >= 1 && !mbar_wait(&o_free[h], (c.sgw - 1) & 1, ERR_WAIT_EPI)) {
            ok = false;
            break;
          }
          // V of this stage: complete (the S of this tile, computed from the same stage, was
          // read before P existed); waiting also makes the TMA writes visible to this thread
          if (!mbar_wait(&kv_full[st], (n / kAttnStages) & 1, ERR_WAIT_TMA)) { ok = false; break; }
          tc_fence_after();
          const uint64_t vdesc =
              sdesc_sw128(smem_u32(sKV + st * L::kStageBytes + L::kKBytes), L::kKVHalf, 1024);
          const uint32_t pa = tmem + 384 + (h * 2 + buf) * 32;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts(tmem + h * 128, pa + kk * 8, vdesc + ((kk * 2048) >> 4), idesc_pv,
                        !(first && kk == 0));
          mma_commit(&o_done[h * 2 + buf]);
          mma_commit(&kv_empty[st]);
          cursor_next(c, p, lo, hi, grp_last);
        }
        if (n > 0) mbar_wait(&o_done[h * 2 + ((n - 1) & 1)], ((n - 1) >> 1) & 1, ERR_WAIT_MMA);
      }
      (void)ok;
    }
    __syncwarp();
  } else {
    // ================================================================ softmax / epilogue
    // Warp w: MMA half h = w / 8, column half c = (w / 4) % 2 (keys 32c..32c+31 of every
    // tile, O columns c*D/2 ..), TMEM lane quarter q4 = w % 4. The two warps (h, 0, q4) and
    // (h, 1, q4) own the same 32 rows: they agree on the row maximum through shared memory and
    // named barrier 1 + 4h + q4, and add their partial row sums at the end of a segment.
    // A wait that runs out records the error and the loop carries on, so both warps of a
    // pair always meet at the same barriers.
    const int h = warp >> 3;
    const int c = (warp >> 2) & 1;
    const int q4 = warp & 3;
    const int rr = q4 * 32 + lane;
    const int r = h * 128 + rr;
    const bool row_ok = r < p.R;
    const bool half_live = h < NH;
    const int bar_id = 1 + h * 4 + q4;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    constexpr int DH = D / 2;
    float* xmax = reinterpret_cast<float*>(smem + L::kOffX);   // [buf][h][c][128]
    float* xl = xmax + 2 * 2 * 2 * 128;                         // [h][c][128]
    const float sc = p.scale_log2;
    int n = 0;
    float m_run = -INFINITY, l_run = 0.f;
    for (int grp = grp_first; grp <= grp_last; ++grp) {
      const SegInfo s = attn_seg(p, lo, hi, grp);
      const int nwork = attn_seg_work(p, s);
      const int s_tok = r / p.Gc;
      const int head = s.g * p.G + s.chunk * p.Gc + (r % p.Gc);
      const int rec = blockIdx.x * p.max_seg + (grp - grp_first);
      if (nwork == 0 || !half_live) {
        // No key reaches this segment (or this half has no rows): an empty partial.
        if (half_live && c == 0 && row_ok && !s.full) {
          p.part_ml[((size_t)rec * p.R + r) * 2 + 0] = -INFINITY;
          p.part_ml[((size_t)rec * p.R + r) * 2 + 1] = 0.f;
        }
        n += nwork;
        continue;
      }
      int wi = 0;
      for (int t = s.t0; t < s.t1; ++t) {
        if (!attn_tile_live(p, s, t)) continue;
        const bool first = (wi == 0), last = (wi == nwork - 1);
        const int buf = n & 1;
        mbar_wait(&s_full[h], n & 1, ERR_WAIT_MMA);
        tc_fence_after();
        float x[32];
        tmem_ld32(tmem + lane_off + 256 + h * 64 + c * 32, x);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&s_empty[h]);
        const int nvalid = (t < p.n_ctx_tiles) ? min(64, s.L - t * 64) : p.S;
        if (nvalid < 64) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c * 32 + j >= nvalid) x[j] = -INFINITY;
        }
        // row maximum of the raw scores (8 independent chains), then the partner's half;
        // scaling by log2(e)/sqrt(D) > 0 commutes with the maximum
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = x[k];
#pragma unroll
        for (int j = 8; j < 32; ++j) mx[j & 7] = fmaxf(mx[j & 7], x[j]);
        const float pm = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        float* xb = xmax + (buf * 2 + h) * 2 * 128;
        xb[c * 128 + rr] = pm;
        pair_sync(bar_id);
        const float tmax = fmaxf(xb[rr], xb[128 + rr]) * sc;
        if (first) {
          m_run = tmax;
          l_run = 0.f;
        } else if (tmax > m_run + 8.0f) {
          const float alpha = ex2_approx(m_run - tmax);
          m_run = tmax;
          l_run *= alpha;
          // every PV so far (the last one used P[(n-1)&1]) must be done before O is touched
          mbar_wait(&o_done[h * 2 + ((n - 1) & 1)], ((n - 1) >> 1) & 1, ERR_WAIT_MMA);
          tc_fence_after();
          const uint32_t oacc = tmem + lane_off + h * 128 + c * DH;
#pragma unroll 1
          for (int k = 0; k < DH / 32; ++k) {
            float o[32];
            tmem_ld32(oacc + k * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] *= alpha;
            tmem_st32(oacc + k * 32, o);
          }
        }
        // P = 2^(x*scale - m) rounded to bf16, two per TMEM column (keys 32c.. -> columns
        // 16c..16c+15 of P[buf]); the running sum adds the fp32 values
        const float mneg = -m_run;
        uint32_t pk[16];
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float e0 = ex2_approx(fmaf(x[2 * j], sc, mneg));
          const float e1 = ex2_approx(fmaf(x[2 * j + 1], sc, mneg));
          pk[j] = pack_bf16x2(e0, e1);
          ls[j & 3] += e0 + e1;
        }
        l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // P[buf] was last read by the PV of tile n-2
        if (n >= 2) mbar_wait(&o_done[h * 2 + buf], ((n - 2) >> 1) & 1, ERR_WAIT_MMA);
        tc_fence_after();
        tmem_st16(tmem + lane_off + 384 + (h * 2 + buf) * 32 + c * 16, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[h * 2 + buf]);
        if (last) {
          mbar_wait(&o_done[h * 2 + buf], (n >> 1) & 1, ERR_WAIT_MMA);
          tc_fence_after();
          // total row sum, added in the same order by both warps of the pair
          xl[(h * 2 + c) * 128 + rr] = l_run;
          pair_sync(bar_id);
          const float ltot = xl[(h * 2) * 128 + rr] + xl[(h * 2 + 1) * 128 + rr];
          const uint32_t oacc = tmem + lane_off + h * 128 + c * DH;
          if (s.full) {
            const float inv = 1.f / ltot;
            uint16_t* dst = p.out + (((size_t)s.b * p.S + s_tok) * p.Hq + head) * D + c * DH;
#pragma unroll 1
            for (int k = 0; k < DH / 32; ++k) {
              float o[32];
              tmem_ld32(oacc + k * 32, o);
              tmem_ld_wait();
              if (row_ok) {
                uint4* d4 = reinterpret_cast<uint4*>(dst + k * 32);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  d4[j] = make_uint4(pack_bf16x2(o[8 * j] * inv, o[8 * j + 1] * inv),
                                     pack_bf16x2(o[8 * j + 2] * inv, o[8 * j + 3] * inv),
                                     pack_bf16x2(o[8 * j + 4] * inv, o[8 * j + 5] * inv),
                                     pack_bf16x2(o[8 * j + 6] * inv, o[8 * j + 7] * inv));
              }
            }
            if (row_ok && c == 0 && p.lse)
              p.lse[((size_t)s.b * p.S + s_tok) * p.Hq + head] =
                  (m_run + __log2f(ltot)) * 0.6931471805599453f;
          } else {
            float* dst = p.part_o + ((size_t)rec * p.R + r) * D + c * DH;
#pragma unroll 1
            for (int k = 0; k < DH / 32; ++k) {
              float o[32];
              tmem_ld32(oacc + k * 32, o);
              tmem_ld_wait();
              if (row_ok) {
                float4* d4 = reinterpret_cast<float4*>(dst + k * 32);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  d4[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
              }
            }
            if (row_ok && c == 0) {
              p.part_ml[((size_t)rec * p.R + r) * 2 + 0] = m_run;
              p.part_ml[((size_t)rec * p.R + r) * 2 + 1] = ltot;
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
  if (warp == kMmaWarp) {
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
