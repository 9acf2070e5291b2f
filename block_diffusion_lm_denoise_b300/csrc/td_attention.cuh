// td_attention.cuh -- fused block attention of the denoiser
// ("NVIDIA、Nemotron-Labs-TwoTowerを公開…", news.chathome.org, inference paragraph: the block
// attends bidirectionally to itself and, layer by layer, to the context tower's KV cache).
//
// Work unit = one (sequence b, KV head g): its S block tokens x G query heads (GQA) read one
// K/V stream. The unit's query rows are cut into NC row chunks of R = S*Gc <= 128 rows (one
// tcgen05 M=128 tile each); a team of NC CTAs, one per chunk, walks the same key range at the
// same pace, so every K/V tile is fetched from HBM once and served to the other CTAs of the
// team from L2. Keys are visited in 128-key tiles: ceil(Lmax/128) context tiles, then one tile
// holding the S block keys; one online softmax runs over all of them (one joint softmax per
// query row). The (unit, tile) space is flattened and cut into equal contiguous ranges, one
// per team (split-K over the context, balanced across the SMs); a CTA whose range covers a
// whole unit writes the normalised bf16 output directly, otherwise it writes an unnormalised
// partial (O, running max, running sum) that attn_merge_kernel combines by log-sum-exp.
//
// Roles (384 threads): warps 0-7 = softmax / epilogue (warp w: TMEM lane quarter w % 4, one
// query row per thread, key half w / 4 = keys 64(w/4)..+63 of every tile and O columns
// (w/4)*D/2..; the two warps of a lane quarter agree on the row maximum through shared
// memory); they also stage the chunk's Q rows into TMEM at each segment start; warps 8, 9
// lane 0 = TMA producers of the K ring and of the V ring (three 32 KB slots each: a K slot is
// recycled as soon as S of its tile is computed, a V slot when PV is); warp 10 lane 0 =
// S = Q K^T issuer (warp 10 also owns the TMEM allocation); warp 11 lane 0 = O += P V issuer.
// TMEM (512 columns): O at 0 (fp32, D columns); S at 128 (fp32, 128 keys); P[buf] at
// 256 + 64 buf (bf16 probabilities, two per column); Q at 384 (bf16, two per column). Both
// MMAs take their A operand (Q, then P) from TMEM, so shared memory holds only K/V tiles and
// serves only B operands. S of tile n+1 is computed as soon as the softmax warps have read
// S(n), i.e. while they work on tile n; P is double buffered, so they never wait on the PV of
// the previous tile. Rescaling of O is lazy: the running max only moves when a tile's max
// exceeds it by more than 8 (log2 units), so P stays <= 2^8 and the TMEM round trip is rare.
#pragma once

#include "td_ptx.cuh"

namespace td {

constexpr int kKeyTile = 128;

struct AttnParams {
  int B, S, Hq, Hkv, D, Lmax;
  int G, Gc, NC, R;          // heads per KV head, heads per chunk, chunks per unit, rows per chunk
  int NCT;                   // CTA pairs per team (pair kernel): ceil(NC / 2)
  int n_ctx_tiles, T;        // ceil(Lmax/128), T = n_ctx_tiles + 1
  int n_units;               // B * Hkv
  int n_teams;               // gridDim.x / NC
  long long total;           // n_units * T
  int max_seg;               // partial-record slots per CTA
  const int* ctx_len;        // [B] or null
  const uint16_t* q;         // [B, S, Hq, D] bf16
  float* part_o;             // [gridDim.x * max_seg][R][D]
  float* part_ml;            // [gridDim.x * max_seg][R][2]  (max in log2 units, sum)
  uint16_t* out;             // [B, S, Hq, D] bf16
  float* lse;                // [B, S, Hq] or null
  float scale_log2;          // log2(e) / sqrt(D)
  const int* skip;           // when non-null and nonzero, return at once
  // paged context cache: when page_table is set, each layer's cache is a pool
  // [n_pages][Hkv][128][D] and logical 128-key tile t of sequence b is page
  // page_table[b * max_pages + t]
  const int* page_table;
  int max_pages, n_pages;
};

constexpr int kKSlots = 3;         // K ring (a slot is freed when S of its tile is done)
constexpr int kVSlots = 4;         // V ring (a slot is freed when PV of its tile is done)
constexpr int kAttnThreads = 384;   // 8 softmax warps + 2 producers + 2 MMA issuers
constexpr int kKProducerWarp = 8;
constexpr int kVProducerWarp = 9;
constexpr int kQkWarp = 10;
constexpr int kPvWarp = 11;

template <int D>
struct AttnSmem {
  static constexpr int kKVHalf = kKeyTile * 128;              // 128 keys x 64 bf16
  static constexpr int kKBytes = kKVHalf * (D / 64);          // one K (or V) tile
  static constexpr int kOffK = 0;                             // K ring
  static constexpr int kOffV = kOffK + kKSlots * kKBytes;     // V ring
  static constexpr int kOffBar = kOffV + kVSlots * kKBytes;
  static constexpr int kBytes = kOffBar + 512 + 1024;
};

__device__ __forceinline__ void pair_sync(int id) {
  asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

__device__ __forceinline__ long long attn_lo(long long team, long long total, int n_teams) {
  return team * total / n_teams;
}

// TMA coordinates (key row, slab) of context tile t of (sequence b, KV head g): a contiguous
// cache is one [Lmax][D] slab per (b, g); a paged cache is one [128][D] slab per (page, g).
// An out-of-range page is flagged and read as zeros (slab -1 is outside the map).
// kPaged is a compile-time choice, so the contiguous kernels carry no paging code.
template <bool kPaged>
__device__ __forceinline__ bool attn_ctx_coords(const AttnParams& p, int b, int g, int t, int& y,
                                                int& z) {
  if constexpr (!kPaged) {
    y = t * kKeyTile;
    z = b * p.Hkv + g;
    return true;
  }
  const int page = p.page_table[(size_t)b * p.max_pages + t];
  y = 0;
  if (page < 0 || page >= p.n_pages) {
    record_error(ERR_BAD_PAGE);
    z = -1;
    return false;
  }
  z = page * p.Hkv + g;
  return true;
}

// One unit's share of a team's tile range.
struct SegInfo {
  int unit;       // b * Hkv + g
  int b, g;
  int t0, t1;     // tile range [t0, t1) of this segment within the unit
  int L;          // valid context length of sequence b
  int nvt;        // context tiles holding valid keys: ceil(L / 128)
  bool full;      // the segment covers the whole unit
};

__device__ __forceinline__ SegInfo attn_seg(const AttnParams& p, long long lo, long long hi,
                                            int unit) {
  SegInfo s;
  s.unit = unit;
  s.b = unit / p.Hkv;
  s.g = unit % p.Hkv;
  const long long base = (long long)unit * p.T;
  s.t0 = (int)((lo > base ? lo : base) - base);
  s.t1 = (int)((hi < base + p.T ? hi : base + p.T) - base);
  s.L = p.ctx_len ? min(max(p.ctx_len[s.b], 0), p.Lmax) : p.Lmax;
  s.nvt = (s.L + kKeyTile - 1) / kKeyTile;
  s.full = (s.t0 == 0 && s.t1 == p.T);
  return s;
}

// The t-th tile of a unit carries work if it is a context tile with valid keys or the block
// tile (t == n_ctx_tiles).
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

// Walks the live tiles of one team's range in order, segment by segment.
struct TileCursor {
  SegInfo s;
  int unit, t, wi, nwork, sgw;   // sgw: index among segments with work
  bool valid;
};

__device__ __forceinline__ void cursor_next_segment(TileCursor& c, const AttnParams& p,
                                                    long long lo, long long hi, int u_last) {
  for (++c.unit; c.unit <= u_last; ++c.unit) {
    const SegInfo s = attn_seg(p, lo, hi, c.unit);
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
                                            long long hi, int u_first, int u_last) {
  c.unit = u_first - 1;
  c.sgw = -1;
  c.valid = false;
  cursor_next_segment(c, p, lo, hi, u_last);
}

__device__ __forceinline__ void cursor_next(TileCursor& c, const AttnParams& p, long long lo,
                                            long long hi, int u_last) {
  if (c.valid && c.wi + 1 < c.nwork) {
    ++c.t;
    while (!attn_tile_live(p, c.s, c.t)) ++c.t;
    ++c.wi;
    return;
  }
  cursor_next_segment(c, p, lo, hi, u_last);
}

// kSplitP: P enters O += P V as two bf16 values (hi = bf16(P) at TMEM columns 256.., lo =
// bf16(P - hi) at 320..) with a second product per key step; P is then single buffered
// (softmax of tile n waits for the P V of tile n - 1).
template <int D, bool kPaged, bool kSplitP>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fused_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmKc,
                      const __grid_constant__ CUtensorMap tmVc,
                      const __grid_constant__ CUtensorMap tmKb,
                      const __grid_constant__ CUtensorMap tmVb, const AttnParams p) {
  using L = AttnSmem<D>;
  if (p.skip != nullptr && *p.skip != 0) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem + L::kOffK;
  uint8_t* sV = smem + L::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* k_full = bars;                        // [K slot]
  uint64_t* k_empty = k_full + kKSlots;           // [K slot]
  uint64_t* v_full = k_empty + kKSlots;           // [V slot]
  uint64_t* v_empty = v_full + kVSlots;           // [V slot]
  uint64_t* q_full = v_empty + kVSlots;           //        Q staged in TMEM
  uint64_t* q_empty = q_full + 1;                 //        last S of a segment done
  uint64_t* s_full = q_full + 2;                  //        S written
  uint64_t* s_free = s_full + 1;                  //        S read by the softmax warps
  uint64_t* p_full = s_free + 1;                  // [buf]  P written
  uint64_t* o_done = p_full + 2;                  // [buf]  PV of a tile that used P[buf] done
  uint64_t* o_free = o_done + 2;                  //        O read out at a segment end
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_free + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int team = blockIdx.x / p.NC;
  const int chunk = blockIdx.x % p.NC;
  const long long lo = attn_lo(team, p.total, p.n_teams);
  const long long hi = attn_lo(team + 1, p.total, p.n_teams);
  const int u_first = (int)(lo / p.T);
  const int u_last = (int)((hi - 1) / p.T);

  // Zero the tiles once: rows that no TMA box covers (padding query rows, block-key rows
  // beyond S) must hold finite values because P = 0 multiplies them.
  {
    uint4* z = reinterpret_cast<uint4*>(smem);
    const int n16 = L::kOffBar / 16;
    for (int i = threadIdx.x; i < n16; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kKSlots; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < kVSlots; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(q_full, 256);
    mbar_init(q_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(s_free, 256);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 256);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(o_free, 256);
    fence_mbar_init();
  }
  if (warp == kQkWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kKProducerWarp || warp == kVProducerWarp) {
    // ================================================================ TMA producers
    // warp 8 fills the K ring, warp 9 the V ring; each walks the same live tiles in order
    const bool is_v = (warp == kVProducerWarp);
    if (lane == 0) {
      const CUtensorMap* mc = is_v ? &tmVc : &tmKc;
      const CUtensorMap* mb = is_v ? &tmVb : &tmKb;
      uint8_t* ring = is_v ? sV : sK;
      uint64_t* full = is_v ? v_full : k_full;
      uint64_t* empty = is_v ? v_empty : k_empty;
      const int nslot = is_v ? kVSlots : kKSlots;
      tma_prefetch_desc(mc);
      tma_prefetch_desc(mb);
      int n = 0;
      bool ok = true;
      for (int u = u_first; u <= u_last && ok; ++u) {
        const SegInfo s = attn_seg(p, lo, hi, u);
        if (attn_seg_work(p, s) == 0) continue;
        for (int t = s.t0; t < s.t1; ++t) {
          if (!attn_tile_live(p, s, t)) continue;
          const int st = n % nslot;
          if (n >= nslot && !mbar_wait(&empty[st], ((n / nslot) & 1) ^ 1, ERR_WAIT_MMA)) {
            ok = false;
            break;
          }
          uint8_t* dst = ring + st * L::kKBytes;
          if (t < p.n_ctx_tiles) {
            int y, z;
            attn_ctx_coords<kPaged>(p, s.b, s.g, t, y, z);
            mbar_arrive_expect_tx(&full[st], kKeyTile * 128 * (D / 64));
            for (int kh = 0; kh < D / 64; ++kh)
              tma_load_3d(dst + kh * L::kKVHalf, mc, &full[st], kh * 64, y, z);
          } else {
            mbar_arrive_expect_tx(&full[st], p.S * 128 * (D / 64));
            for (int kh = 0; kh < D / 64; ++kh)
              tma_load_4d(dst + kh * L::kKVHalf, mb, &full[st], kh * 64, s.g, 0, s.b);
          }
          ++n;
        }
      }
      if (!ok) {
        for (int j = (n > nslot ? n - nslot : 0); j < n; ++j)
          mbar_wait_drain(&full[j % nslot], (j / nslot) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kQkWarp) {
    // ================================================================ S = Q K^T issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, kKeyTile, 0);
      TileCursor c;
      cursor_init(c, p, lo, hi, u_first, u_last);
      int n = 0;
      for (; c.valid; ++n) {
        const int st = n % kKSlots;
        if (!mbar_wait(&k_full[st], (n / kKSlots) & 1, ERR_WAIT_TMA)) break;
        if (c.wi == 0 && !mbar_wait(q_full, c.sgw & 1, ERR_WAIT_EPI)) break;
        if (n >= 1 && !mbar_wait(s_free, (n - 1) & 1, ERR_WAIT_EPI)) break;
        tc_fence_after();
        // descriptor of k-step 0; later k-steps add (byte offset >> 4) to the address field
        const uint64_t kdesc = sdesc_sw128(smem_u32(sK + st * L::kKBytes), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t kb = kdesc + (((kk >> 2) * L::kKVHalf + (kk & 3) * 32) >> 4);
          mma_bf16_ts(tmem + 128, tmem + 384 + kk * 8, kb, idesc_qk, kk != 0);
        }
        mma_commit(s_full);
        mma_commit(&k_empty[st]);
        if (c.wi == c.nwork - 1) mma_commit(q_empty);
        cursor_next(c, p, lo, hi, u_last);
      }
      // Let every MMA issued so far finish before the TMEM is released.
      if (n > 0) mbar_wait_drain(s_full, (n - 1) & 1);
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ================================================================ O += P V issuer
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, 1);
      TileCursor c;
      cursor_init(c, p, lo, hi, u_first, u_last);
      int n = 0;
      for (; c.valid; ++n) {
        const int st = n % kVSlots;
        const int buf = n & 1;
        const bool first = c.wi == 0;
        if (!mbar_wait(&p_full[buf], (n >> 1) & 1, ERR_WAIT_EPI)) break;
        if (first && c.sgw >= 1 && !mbar_wait(o_free, (c.sgw - 1) & 1, ERR_WAIT_EPI)) break;
        if (!mbar_wait(&v_full[st], (n / kVSlots) & 1, ERR_WAIT_TMA)) break;
        tc_fence_after();
        const uint64_t vdesc = sdesc_sw128(smem_u32(sV + st * L::kKBytes), L::kKVHalf, 1024);
        const uint32_t pa = tmem + 256 + (kSplitP ? 0 : buf * 64);
#pragma unroll
        for (int kk = 0; kk < kKeyTile / 16; ++kk)
          mma_bf16_ts(tmem, pa + kk * 8, vdesc + ((kk * 2048) >> 4), idesc_pv,
                      !(first && kk == 0));
        if constexpr (kSplitP) {
#pragma unroll
          for (int kk = 0; kk < kKeyTile / 16; ++kk)
            mma_bf16_ts(tmem, pa + 64 + kk * 8, vdesc + ((kk * 2048) >> 4), idesc_pv, 1);
        }
        mma_commit(&o_done[buf]);
        mma_commit(&v_empty[st]);
        cursor_next(c, p, lo, hi, u_last);
      }
      if (n > 0) mbar_wait_drain(&o_done[(n - 1) & 1], ((n - 1) >> 1) & 1);
    }
    __syncwarp();
  } else {
    // ================================================================ softmax / epilogue
    // Warp w (0..7): TMEM lane quarter q4 = w % 4 (thread i holds query row 32 q4 + i), key
    // half kh = w / 4 (keys 64 kh .. 64 kh + 63 of every tile, O columns kh*D/2 ..). The two
    // warps of a lane quarter agree on each tile's row maximum through TMEM columns 448..
    // (both can address their lane quarter) and named barrier 1 + q4, and add their partial
    // row sums at the end of a segment. At each
    // segment start they stage their rows of Q into TMEM. A wait that runs out records the
    // error and the loop carries on, so both warps of a pair always meet at the same barriers.
    const int q4 = warp & 3;
    const int kh = warp >> 2;
    const int r = q4 * 32 + lane;
    const bool row_ok = r < p.R;
    const int bar_id = 1 + q4;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    constexpr int DH = D / 2;                                    // O columns of this warp
    // exchange columns: row max of tile n at 448 + 2(n&1) + kh, row sums at 452 + kh
    const uint32_t xcol = tmem + lane_off + 448;
    const float sc = p.scale_log2;
    const int s_tok = r / p.Gc;
    int n = 0, sgw = 0;
    float m_run = -INFINITY, l_run = 0.f;
    for (int u = u_first; u <= u_last; ++u) {
      const SegInfo s = attn_seg(p, lo, hi, u);
      const int nwork = attn_seg_work(p, s);
      const int head = s.g * p.G + chunk * p.Gc + (r % p.Gc);
      const int rec = blockIdx.x * p.max_seg + (u - u_first);
      if (nwork == 0) {
        // No key reaches this segment: an empty partial.
        if (kh == 0 && row_ok && !s.full) {
          p.part_ml[((size_t)rec * p.R + r) * 2 + 0] = -INFINITY;
          p.part_ml[((size_t)rec * p.R + r) * 2 + 1] = 0.f;
        }
        continue;
      }
      {
        // Stage this row's half of Q (elements kh*D/2 ..) into TMEM columns 384 + kh*D/4 ..,
        // once the last S of the previous segment has been computed.
        if (sgw >= 1) mbar_wait(q_empty, (sgw - 1) & 1, ERR_WAIT_MMA);
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + (((size_t)s.b * p.S + s_tok) * p.Hq + head) * D + kh * DH);
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < DH / 32; ++k) {
          uint32_t qv[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 w = row_ok ? __ldg(&src[4 * k + j]) : make_uint4(0, 0, 0, 0);
            qv[4 * j] = w.x; qv[4 * j + 1] = w.y; qv[4 * j + 2] = w.z; qv[4 * j + 3] = w.w;
          }
          tmem_st16(tmem + lane_off + 384 + kh * (D / 4) + k * 16, qv);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(q_full);
        ++sgw;
      }
      int wi = 0;
      for (int t = s.t0; t < s.t1; ++t) {
        if (!attn_tile_live(p, s, t)) continue;
        const bool first = (wi == 0), last = (wi == nwork - 1);
        const int buf = n & 1;
        mbar_wait(s_full, n & 1, ERR_WAIT_MMA);
        tc_fence_after();
        float x[64];
        {
          float (&x0)[32] = *reinterpret_cast<float (*)[32]>(&x[0]);
          float (&x1)[32] = *reinterpret_cast<float (*)[32]>(&x[32]);
          tmem_ld32(tmem + lane_off + 128 + kh * 64, x0);
          tmem_ld32(tmem + lane_off + 128 + kh * 64 + 32, x1);
        }
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(s_free);
        const int nvalid = (t < p.n_ctx_tiles) ? min(kKeyTile, s.L - t * kKeyTile) : p.S;
        if (nvalid < kKeyTile) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (kh * 64 + j >= nvalid) x[j] = -INFINITY;
        }
        // row maximum of the raw scores (8 independent chains), then the partner's half;
        // scaling by log2(e)/sqrt(D) > 0 commutes with the maximum
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = x[k];
#pragma unroll
        for (int j = 8; j < 64; ++j) mx[j & 7] = fmaxf(mx[j & 7], x[j]);
        const float pmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        tmem_st1(xcol + 2 * buf + kh, pmax);
        tmem_st_wait();
        tc_fence_before();
        pair_sync(bar_id);
        tc_fence_after();
        const float omax = tmem_ld1(xcol + 2 * buf + (1 - kh));
        tmem_ld_wait();
        const float tmax = fmaxf(pmax, omax) * sc;
        if (first) {
          m_run = tmax;
          l_run = 0.f;
        } else if (tmax > m_run + 8.0f) {
          const float alpha = ex2_approx(m_run - tmax);
          m_run = tmax;
          l_run *= alpha;
          // every PV so far (the last one used P[(n-1)&1]) must be done before O is touched
          mbar_wait(&o_done[(n - 1) & 1], ((n - 1) >> 1) & 1, ERR_WAIT_MMA);
          tc_fence_after();
#pragma unroll 1
          for (int k = 0; k < DH / 32; ++k) {
            float o[32];
            tmem_ld32(tmem + lane_off + kh * DH + 32 * k, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] *= alpha;
            tmem_st32(tmem + lane_off + kh * DH + 32 * k, o);
          }
        }
        // P[buf] was last read by the PV of tile n-2 (split P: the one P area by tile n-1)
        if constexpr (kSplitP) {
          if (n >= 1) mbar_wait(&o_done[(n - 1) & 1], ((n - 1) >> 1) & 1, ERR_WAIT_MMA);
        } else {
          if (n >= 2) mbar_wait(&o_done[buf], ((n - 2) >> 1) & 1, ERR_WAIT_MMA);
        }
        tc_fence_after();
        // P = 2^(x*scale - m) rounded to bf16, two per TMEM column (keys 64kh.. -> columns
        // 32kh.. of P[buf]); the running sum adds the fp32 values
        const float mneg = -m_run;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          uint32_t pk[16], pl[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float e0 = ex2_approx(fmaf(x[32 * k + 2 * j], sc, mneg));
            const float e1 = ex2_approx(fmaf(x[32 * k + 2 * j + 1], sc, mneg));
            pk[j] = pack_bf16x2(e0, e1);
            if constexpr (kSplitP)
              pl[j] = pack_bf16x2(e0 - bf16lo_to_f32(pk[j]), e1 - bf16hi_to_f32(pk[j]));
            ls[j & 3] += e0 + e1;
          }
          const uint32_t pcol = 256 + (kSplitP ? 0 : buf * 64) + kh * 32 + 16 * k;
          tmem_st16(tmem + lane_off + pcol, pk);
          if constexpr (kSplitP) tmem_st16(tmem + lane_off + pcol + 64, pl);
        }
        l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[buf]);
        if (last) {
          mbar_wait(&o_done[buf], (n >> 1) & 1, ERR_WAIT_MMA);
          tc_fence_after();
          // total row sum, added in the same order (half 0 + half 1) by both warps
          tmem_st1(xcol + 4 + kh, l_run);
          tmem_st_wait();
          tc_fence_before();
          pair_sync(bar_id);
          tc_fence_after();
          const float lo_other = tmem_ld1(xcol + 4 + (1 - kh));
          tmem_ld_wait();
          const float ltot = kh == 0 ? l_run + lo_other : lo_other + l_run;
          const float inv = 1.f / ltot;
#pragma unroll 1
          for (int k = 0; k < DH / 32; ++k) {
            float o[32];
            tmem_ld32(tmem + lane_off + kh * DH + 32 * k, o);
            tmem_ld_wait();
            if (!row_ok) continue;
            if (s.full) {
              uint4* d4 = reinterpret_cast<uint4*>(
                  p.out + (((size_t)s.b * p.S + s_tok) * p.Hq + head) * D + kh * DH + 32 * k);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                d4[j] = make_uint4(pack_bf16x2(o[8 * j] * inv, o[8 * j + 1] * inv),
                                   pack_bf16x2(o[8 * j + 2] * inv, o[8 * j + 3] * inv),
                                   pack_bf16x2(o[8 * j + 4] * inv, o[8 * j + 5] * inv),
                                   pack_bf16x2(o[8 * j + 6] * inv, o[8 * j + 7] * inv));
            } else {
              float4* d4 = reinterpret_cast<float4*>(p.part_o + ((size_t)rec * p.R + r) * D +
                                                     kh * DH + 32 * k);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                d4[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            }
          }
          if (row_ok && kh == 0) {
            if (s.full) {
              if (p.lse)
                p.lse[((size_t)s.b * p.S + s_tok) * p.Hq + head] =
                    (m_run + __log2f(ltot)) * 0.6931471805599453f;
            } else {
              p.part_ml[((size_t)rec * p.R + r) * 2 + 0] = m_run;
              p.part_ml[((size_t)rec * p.R + r) * 2 + 1] = ltot;
            }
          }
          tc_fence_before();
          mbar_arrive(o_free);
        }
        ++n;
        ++wi;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kQkWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Log-sum-exp merge of the partials of every (unit, row chunk) that no single team covered.
// Grid: (unit, chunk) x ceil(R / kMergeRows) row groups; thread (row, 4 columns). One thread
// per CTA finds the teams that share the unit and their record indices (64-bit integer
// arithmetic, done once instead of by every thread) and hands them over in shared memory.
constexpr int kMergeRows = 16;
constexpr int kMergeTeams = 16;   // teams per unit handled per pass of the record loop

// The team whose key range holds (unit, tile) index x: the largest k with lo(k) <= x, i.e.
// k * total < (x + 1) * n_teams.
__device__ __forceinline__ int attn_owner(long long x, long long total, int n_teams) {
  const long long k = ((x + 1) * n_teams - 1) / total;
  return (int)(k < n_teams - 1 ? k : n_teams - 1);
}

__global__ void __launch_bounds__(512) attn_merge_kernel(const AttnParams p) {
  if (p.skip != nullptr && *p.skip != 0) return;
  __shared__ int s_k[2];
  __shared__ int s_rec[kMergeTeams];
  const int uc = blockIdx.x;
  const int unit = uc / p.NC;
  const int chunk = uc % p.NC;
  if (threadIdx.x == 0) {
    const long long first_tile = (long long)unit * p.T;
    s_k[0] = attn_owner(first_tile, p.total, p.n_teams);
    s_k[1] = attn_owner(first_tile + p.T - 1, p.total, p.n_teams);
  }
  __syncthreads();
  const int k0 = s_k[0];
  const int k1 = s_k[1];
  if (k0 == k1) return;   // written directly by its only team
  const int b = unit / p.Hkv;
  const int g = unit % p.Hkv;
  const int D = p.D;
  const int nq4 = D / 4;
  const int r = blockIdx.y * kMergeRows + threadIdx.x / nq4;
  // threads past the rows stay for the barriers of the record loop
  const bool row_ok = threadIdx.x < kMergeRows * nq4 && r < p.R;
  const int d4 = threadIdx.x % nq4;
  // the teams' records, kMergeTeams at a time; maximum first, then the weighted sums, both
  // over the teams in order
  float M = -INFINITY;
  float Lsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int pass = 0; pass < 2; ++pass) {
    for (int kb = k0; kb <= k1; kb += kMergeTeams) {
      const int nk = min(kMergeTeams, k1 - kb + 1);
      __syncthreads();
      if (threadIdx.x < nk)
        s_rec[threadIdx.x] =
            ((kb + threadIdx.x) * p.NC + chunk) * p.max_seg +
            (unit - (int)(attn_lo(kb + threadIdx.x, p.total, p.n_teams) / p.T));
      __syncthreads();
      if (!row_ok) continue;
      for (int i = 0; i < nk; ++i) {
        const size_t rr = (size_t)s_rec[i] * p.R + r;
        const float mk = __ldg(&p.part_ml[rr * 2]);
        if (pass == 0) {
          M = fmaxf(M, mk);
          continue;
        }
        const float lk = __ldg(&p.part_ml[rr * 2 + 1]);
        if (lk == 0.f) continue;
        const float w = exp2f(mk - M);
        Lsum += lk * w;
        const float4 o = __ldg(reinterpret_cast<const float4*>(p.part_o + rr * D) + d4);
        acc.x += o.x * w; acc.y += o.y * w; acc.z += o.z * w; acc.w += o.w * w;
      }
    }
  }
  if (!row_ok) return;
  const float inv = 1.f / Lsum;
  const int s_tok = r / p.Gc;
  const int head = g * p.G + chunk * p.Gc + (r % p.Gc);
  uint16_t* dst = p.out + (((size_t)b * p.S + s_tok) * p.Hq + head) * D + d4 * 4;
  *reinterpret_cast<uint2*>(dst) =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (d4 == 0 && p.lse)
    p.lse[((size_t)b * p.S + s_tok) * p.Hq + head] = (M + log2f(Lsum)) * 0.6931471805599453f;
}

}  // namespace td
