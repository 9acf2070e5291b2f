// td_attention_pair.cuh -- the fused block attention on SM pairs (head_dim 128)
// ("NVIDIA、Nemotron-Labs-TwoTowerを公開…", news.chathome.org, inference paragraph: the block
// attends bidirectionally to itself and, layer by layer, to the context tower's KV cache).
//
// Same work split, tiles and online softmax as attn_fused_kernel, but the two 128-row chunks
// of a unit sit on the two SMs of one TPC (a cluster of two CTAs) and every product is one
// tcgen05 pair MMA (cta_group::2, M = 256) issued by the even CTA:
//   S  = Q K^T : A = each CTA's Q chunk (shared memory), B = K tile split by keys (CTA r holds
//                keys 64r..64r+63 of the 128-key tile), D = each CTA's 128 x 128 scores;
//   O += P V   : A = each CTA's P (TMEM), B = V tile split by columns (CTA r holds head
//                dimensions 64r..64r+63 of all 128 keys), D = each CTA's 128 x 128 O (TMEM).
// So each SM streams only half of every K/V tile from L2/HBM into its shared memory, and one
// MMA instruction serves 256 query rows.
//
// Scores live in three TMEM buffers SP[b] (tile n uses SP[n % 3]): S in fp32, then P in bf16
// pairs over its first 64 columns once both warps of a lane quarter have read their S. The S
// product of tile n waits only for the O += P V of tile n - 3 (the last reader of its
// buffer), which keeps the chain S(n) -> softmax(n) -> O += P V(n) -> S(n + 3) off the
// critical path: the softmax warps find the next S ready when they finish a tile.
//
// Barriers that gate the MMAs (K/V/Q landed, P written, O read out) live in the even CTA: the
// odd CTA's TMA loads complete their bytes there (cp.async.bulk.tensor .cta_group::2) and its
// softmax warps arrive there through the cluster window. Barriers that the MMAs release
// (S ready, O updated, ring slots free, Q consumed) exist in both CTAs and are signalled by
// one multicast commit.
//
// Roles per CTA (384 threads): warps 0-7 = softmax / epilogue (warp w: TMEM lane quarter
// w % 4, key half w / 4; the two warps of a lane quarter agree on the row maximum through
// shared memory and a named barrier); warp 8 lane 0 = producer of the K ring and of each
// segment's Q, warp 9 lane 0 = producer of the V ring (each CTA loads its own halves);
// warp 10 owns the TMEM (allocated for the pair) and, in the even CTA, lane 0 issues
// S = Q K^T; warp 11 lane 0 of the even CTA issues O += P V. TMEM per CTA: O at 0, SP[b] at
// 128 + 128 b.
#pragma once

#include "td_attention.cuh"

namespace td {

constexpr int kPairKSlots = 5;      // K ring: 16 KB slots (64 keys x 128 dims)
constexpr int kPairVSlots = 6;      // V ring: 16 KB slots (128 keys x 64 dims)
constexpr int kPairSP = 3;          // score / probability buffers in TMEM

struct PairSmem {
  static constexpr int kKHalf = 64 * 128;                     // 64 keys x 64 dims
  static constexpr int kKBytes = 2 * kKHalf;                  // one K slot
  static constexpr int kVBytes = kKeyTile * 128;              // one V slot (128 keys x 64 dims)
  static constexpr int kQHalf = 128 * 128;                    // 128 rows x 64 dims
  static constexpr int kOffQ = 0;                             // Q chunk (A operand), 32 KB
  static constexpr int kOffK = kOffQ + 2 * kQHalf;
  static constexpr int kOffV = kOffK + kPairKSlots * kKBytes;
  static constexpr int kOffX = kOffV + kPairVSlots * kVBytes; // row max / sum exchange
  static constexpr int kXFloats = 3 * 2 * 128;                // [max tile n & 1 | sum][kh][row]
  static constexpr int kOffBar = kOffX + kXFloats * 4;
  static constexpr int kBytes = kOffBar + 512 + 1024;
};

// The O readout at the end of a segment, out of line: it runs once per segment, and inline it
// would sit in the per-tile loop's code.
__device__ __noinline__ void pair_epilogue(uint16_t* out, float* part_o, float* part_ml, float* lse,
                                           int S, int Hq, int R, uint32_t tmem, uint32_t lane_off,
                                           int kh, int r, bool row_ok, float* xch, int bar_id,
                                           uint64_t* o_done_bar, uint32_t parity,
                                           uint64_t* o_free, bool even, int lane, float m_run,
                                           float l_run, bool full, int b, int s_tok, int head,
                                           size_t rec) {
  constexpr int D = 128;
  constexpr int DH = D / 2;
  mbar_wait(o_done_bar, parity, ERR_WAIT_MMA);
  tc_fence_after();
  float* xl = xch + 512;
  xl[kh * 128 + r] = l_run;
  pair_sync(bar_id);
  const float lo_other = xl[(1 - kh) * 128 + r];
  const float ltot = kh == 0 ? l_run + lo_other : lo_other + l_run;
  const float inv = 1.f / ltot;
#pragma unroll 1
  for (int k = 0; k < DH / 32; ++k) {
    float o[32];
    tmem_ld32(tmem + lane_off + kh * DH + 32 * k, o);
    tmem_ld_wait();
    if (!row_ok) continue;
    if (full) {
      uint4* d4 = reinterpret_cast<uint4*>(out +
                                           (((size_t)b * S + s_tok) * Hq + head) * D + kh * DH +
                                           32 * k);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        d4[j] = make_uint4(pack_bf16x2(o[8 * j] * inv, o[8 * j + 1] * inv),
                           pack_bf16x2(o[8 * j + 2] * inv, o[8 * j + 3] * inv),
                           pack_bf16x2(o[8 * j + 4] * inv, o[8 * j + 5] * inv),
                           pack_bf16x2(o[8 * j + 6] * inv, o[8 * j + 7] * inv));
    } else {
      float4* d4 = reinterpret_cast<float4*>(part_o + (rec * R + r) * D + kh * DH + 32 * k);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        d4[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
    }
  }
  if (row_ok && kh == 0) {
    if (full) {
      if (lse)
        lse[((size_t)b * S + s_tok) * Hq + head] = (m_run + __log2f(ltot)) * 0.6931471805599453f;
    } else {
      part_ml[(rec * R + r) * 2 + 0] = m_run;
      part_ml[(rec * R + r) * 2 + 1] = ltot;
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    if (even) mbar_arrive(o_free);
    else mbar_arrive_cluster_relaxed(cluster_addr(o_free, 0));
  }
}

// Lazy rescale of this warp's O columns by alpha, out of line (rare).
__device__ __noinline__ void pair_rescale(uint32_t tmem, uint32_t lane_off, int kh, float alpha,
                                          uint64_t* o_done_bar, uint32_t parity) {
  constexpr int DH = 64;
  mbar_wait(o_done_bar, parity, ERR_WAIT_MMA);
  tc_fence_after();
#pragma unroll 1
  for (int k = 0; k < DH / 8; ++k) {
    uint32_t o[8];
    tmem_ld8(tmem + lane_off + kh * DH + 8 * k, o);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
    tmem_st8(tmem + lane_off + kh * DH + 8 * k, o);
  }
}

// kSplitP: P enters O += P V as two bf16 values, hi = bf16(P) over the first 64 columns of
// SP[buf] and lo = bf16(P - hi) over the other 64 (both warps of a lane quarter have read
// their scores by then), with a second product per key step: P is then carried to about
// 2^-17 relative instead of 2^-9.
template <bool kPaged, bool kSplitP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttnThreads, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmKc,
                     const __grid_constant__ CUtensorMap tmVc,
                     const __grid_constant__ CUtensorMap tmKb,
                     const __grid_constant__ CUtensorMap tmVb, const AttnParams p) {
  constexpr int D = 128;
  using L = PairSmem;
  if (p.skip != nullptr && *p.skip != 0) return;   // both CTAs of a pair read the same flag
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sK = smem + L::kOffK;
  uint8_t* sV = smem + L::kOffV;
  float* xch = reinterpret_cast<float*>(smem + L::kOffX);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  // gating barriers, used in the even CTA
  uint64_t* k_full = bars;                        // [K slot] both halves landed
  uint64_t* v_full = k_full + kPairKSlots;        // [V slot]
  uint64_t* q_full = v_full + kPairVSlots;        //          both Q chunks landed
  uint64_t* p_full = q_full + 1;                  // [buf]    P written in both CTAs
  uint64_t* o_free = p_full + kPairSP;            //          O read out in both CTAs
  // barriers signalled by the MMAs in both CTAs
  uint64_t* k_empty = o_free + 1;                 // [K slot]
  uint64_t* v_empty = k_empty + kPairKSlots;      // [V slot]
  uint64_t* q_empty = v_empty + kPairVSlots;      //          last S of a segment done
  uint64_t* s_full = q_empty + 1;                 // [buf]    S written into SP[buf]
  uint64_t* o_done = s_full + kPairSP;            // [buf]    O += P V with SP[buf] done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_done + kPairSP);

  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x >> 1;
  const int team = pair / p.NCT;
  const int chunk = 2 * (pair % p.NCT) + (int)rank;
  const bool chunk_ok = chunk < p.NC;
  const long long lo = attn_lo(team, p.total, p.n_teams);
  const long long hi = attn_lo(team + 1, p.total, p.n_teams);
  const int u_first = (int)(lo / p.T);
  const int u_last = (int)((hi - 1) / p.T);

  // Q rows beyond R are never loaded: they must hold finite values (zeros)
  {
    uint4* z = reinterpret_cast<uint4*>(sQ);
    for (int i = threadIdx.x; i < 2 * L::kQHalf / 16; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPairKSlots; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < kPairVSlots; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(o_free, 16);          // 8 softmax warps x 2 CTAs
    for (int i = 0; i < kPairSP; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 16);
      mbar_init(&o_done[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == kQkWarp) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before any cross-CTA arrival or byte count
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kKProducerWarp || warp == kVProducerWarp) {
    // ================================================================ TMA producers
    const bool is_v = (warp == kVProducerWarp);
    if (lane == 0) {
      const CUtensorMap* mc = is_v ? &tmVc : &tmKc;
      const CUtensorMap* mb = is_v ? &tmVb : &tmKb;
      uint8_t* ring = is_v ? sV : sK;
      uint64_t* full = is_v ? v_full : k_full;
      uint64_t* empty = is_v ? v_empty : k_empty;
      const int nslot = is_v ? kPairVSlots : kPairKSlots;
      const int slot_bytes = is_v ? L::kVBytes : L::kKBytes;
      // this CTA's half of a tile: K rows 64r.. (both dim halves), V dims 64r..
      const int kx = is_v ? 64 * (int)rank : 0;
      const int ky = is_v ? 0 : 64 * (int)rank;
      const uint32_t q_bytes = 2u * 2u * (uint32_t)p.R * 128u;   // 2 CTAs x 2 dim halves
      tma_prefetch_desc(mc);
      tma_prefetch_desc(mb);
      if (!is_v) tma_prefetch_desc(&tmQ);
      int n = 0, sg = 0;
      bool ok = true;
      for (int u = u_first; u <= u_last && ok; ++u) {
        const SegInfo s = attn_seg(p, lo, hi, u);
        if (attn_seg_work(p, s) == 0) continue;
        bool q_pending = !is_v;
        if (q_pending && sg == 0) {
          // the first Q goes out before the ring fills
          q_pending = false;
          if (even) mbar_arrive_expect_tx(q_full, q_bytes);
          for (int kh = 0; kh < 2; ++kh)
            tma_load_4d_pair(sQ + kh * L::kQHalf, &tmQ, cluster_addr(q_full, 0), kh * 64,
                             s.g * p.G + chunk * p.Gc, 0, s.b);
          ++sg;
        }
        for (int t = s.t0; t < s.t1; ++t) {
          if (!attn_tile_live(p, s, t)) continue;
          const int st = n % nslot;
          if (n >= nslot && !mbar_wait(&empty[st], ((n / nslot) & 1) ^ 1, ERR_WAIT_MMA)) {
            ok = false;
            break;
          }
          const uint32_t bar = cluster_addr(&full[st], 0);
          if (even) mbar_arrive_expect_tx(&full[st], 2 * slot_bytes);   // both CTAs' halves
          uint8_t* dst = ring + st * slot_bytes;
          if (t < p.n_ctx_tiles) {
            int y, z;
            attn_ctx_coords<kPaged>(p, s.b, s.g, t, y, z);
            if (is_v) tma_load_3d_pair(dst, mc, bar, kx, y, z);
            else
              for (int kh = 0; kh < 2; ++kh)
                tma_load_3d_pair(dst + kh * L::kKHalf, mc, bar, kh * 64, y + ky, z);
          } else {
            // the block keys: rows beyond S are out of bounds and arrive as zeros
            if (is_v) tma_load_4d_pair(dst, mb, bar, kx, s.g, 0, s.b);
            else
              for (int kh = 0; kh < 2; ++kh)
                tma_load_4d_pair(dst + kh * L::kKHalf, mb, bar, kh * 64, s.g, ky, s.b);
          }
          ++n;
          if (q_pending) {
            // this CTA's Q chunk (rows s * Gc + head-in-chunk), once the last S product of
            // the previous segment has read the old one
            q_pending = false;
            if (sg >= 1 && !mbar_wait(q_empty, (sg - 1) & 1, ERR_WAIT_MMA)) {
              ok = false;
              break;
            }
            const uint32_t qbar = cluster_addr(q_full, 0);
            if (even) mbar_arrive_expect_tx(q_full, q_bytes);
            for (int kh = 0; kh < 2; ++kh)
              tma_load_4d_pair(sQ + kh * L::kQHalf, &tmQ, qbar, kh * 64, s.g * p.G + chunk * p.Gc,
                               0, s.b);
            ++sg;
          }
        }
      }
      if (!ok && even) {
        // let the copies in flight land before the kernel returns
        for (int j = (n > nslot ? n - nslot : 0); j < n; ++j)
          mbar_wait_drain(&full[j % nslot], (j / nslot) & 1);
        if (!is_v && sg >= 1) mbar_wait_drain(q_full, (sg - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kQkWarp) {
    // ================================================================ S = Q K^T issuer
    if (even && lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(256, kKeyTile, 0);
      const uint64_t qdesc = sdesc_sw128(smem_u32(sQ), 16, 1024);
      TileCursor c;
      cursor_init(c, p, lo, hi, u_first, u_last);
      int n = 0;
      for (; c.valid; ++n) {
        const int st = n % kPairKSlots;
        const int buf = n % kPairSP;
        if (!mbar_wait(&k_full[st], (n / kPairKSlots) & 1, ERR_WAIT_TMA)) break;
        if (c.wi == 0 && !mbar_wait(q_full, c.sgw & 1, ERR_WAIT_TMA)) break;
        // SP[buf] was last read by the O += P V of tile n - 3
        if (n >= kPairSP &&
            !mbar_wait(&o_done[buf], ((n - kPairSP) / kPairSP) & 1, ERR_WAIT_MMA))
          break;
        tc_fence_after();
        const uint64_t kdesc = sdesc_sw128(smem_u32(sK + st * L::kKBytes), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qo = (uint32_t)(((kk >> 2) * L::kQHalf + (kk & 3) * 32) >> 4);
          const uint32_t ko = (uint32_t)(((kk >> 2) * L::kKHalf + (kk & 3) * 32) >> 4);
          mma_pair_ss(tmem + 128 + 128 * buf, qdesc + qo, kdesc + ko, idesc_qk, kk != 0);
        }
        mma_commit_pair(&s_full[buf], 3);
        mma_commit_pair(&k_empty[st], 3);
        if (c.wi == c.nwork - 1) mma_commit_pair(q_empty, 3);
        cursor_next(c, p, lo, hi, u_last);
      }
      // every MMA issued so far completes before the TMEM is released
      if (n > 0) mbar_wait_drain(&s_full[(n - 1) % kPairSP], ((n - 1) / kPairSP) & 1);
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ================================================================ O += P V issuer
    if (even && lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16(256, D, 1);
      TileCursor c;
      cursor_init(c, p, lo, hi, u_first, u_last);
      int n = 0;
      for (; c.valid; ++n) {
        const int st = n % kPairVSlots;
        const int buf = n % kPairSP;
        const bool first = c.wi == 0;
        const int nvalid =
            c.t < p.n_ctx_tiles ? min(kKeyTile, c.s.L - c.t * kKeyTile) : p.S;
        const int nk = (nvalid + 15) / 16;
        if (!mbar_wait(&p_full[buf], (n / kPairSP) & 1, ERR_WAIT_EPI)) break;
        if (first && c.sgw >= 1 && !mbar_wait(o_free, (c.sgw - 1) & 1, ERR_WAIT_EPI)) break;
        if (!mbar_wait(&v_full[st], (n / kPairVSlots) & 1, ERR_WAIT_TMA)) break;
        tc_fence_after();
        // one 64-column swizzle atom of V per CTA: the leading byte offset is not used
        const uint64_t vdesc = sdesc_sw128(smem_u32(sV + st * L::kVBytes), L::kVBytes, 1024);
        const uint32_t pa = tmem + 128 + 128 * buf;
        // a full tile's eight products go out as straight-line code: a branch between two
        // tcgen05.mma instructions costs the issuing thread about 100 cycles, more than the
        // 64 the tensor pipe needs for one product
        if (nk == kKeyTile / 16) {
#pragma unroll
          for (int kk = 0; kk < kKeyTile / 16; ++kk)
            mma_pair_ts(tmem, pa + kk * 8, vdesc + ((kk * 2048) >> 4), idesc_pv,
                        !(first && kk == 0));
          if constexpr (kSplitP) {
#pragma unroll
            for (int kk = 0; kk < kKeyTile / 16; ++kk)
              mma_pair_ts(tmem, pa + 64 + kk * 8, vdesc + ((kk * 2048) >> 4), idesc_pv, 1);
          }
        } else {
          for (int kk = 0; kk < nk; ++kk)
            mma_pair_ts(tmem, pa + kk * 8, vdesc + ((kk * 2048) >> 4), idesc_pv,
                        !(first && kk == 0));
          if constexpr (kSplitP)
            for (int kk = 0; kk < nk; ++kk)
              mma_pair_ts(tmem, pa + 64 + kk * 8, vdesc + ((kk * 2048) >> 4), idesc_pv, 1);
        }
        mma_commit_pair(&o_done[buf], 3);
        mma_commit_pair(&v_empty[st], 3);
        cursor_next(c, p, lo, hi, u_last);
      }
      if (n > 0) mbar_wait_drain(&o_done[(n - 1) % kPairSP], ((n - 1) / kPairSP) & 1);
    }
    __syncwarp();
  } else {
    // ================================================================ softmax / epilogue
    // Warp w (0..7): TMEM lane quarter q4 = w % 4 (thread i holds query row 32 q4 + i), key
    // half kh = w / 4 (keys 64 kh .. 64 kh + 63 of every tile, O columns kh*D/2 ..). A wait
    // that runs out records the error and the loop carries on, so both warps of a lane
    // quarter always meet at the same named barriers.
    const int q4 = warp & 3;
    const int kh = warp >> 2;
    const int r = q4 * 32 + lane;
    const bool row_ok = chunk_ok && r < p.R;
    const int bar_id = 1 + q4;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    // hand-off to the even CTA's gating barriers: a local release arrive there, a relaxed
    // arrive through the cluster window from the odd CTA (each follows a completed
    // tcgen05.wait::ld / ::st and tcgen05.fence::before_thread_sync)
    auto hand_off = [&](uint64_t* bar) {
      __syncwarp();
      if (lane == 0) {
        if (even) mbar_arrive(bar);
        else mbar_arrive_cluster_relaxed(cluster_addr(bar, 0));
      }
    };
    const float sc = p.scale_log2;
    const int s_tok = r / p.Gc;
    int n = 0;
    float m_run = -INFINITY, l_run = 0.f;
    for (int u = u_first; u <= u_last; ++u) {
      const SegInfo s = attn_seg(p, lo, hi, u);
      const int nwork = attn_seg_work(p, s);
      const int head = s.g * p.G + chunk * p.Gc + (r % p.Gc);
      const size_t rec = ((size_t)team * p.NC + chunk) * p.max_seg + (u - u_first);
      if (nwork == 0) {
        if (kh == 0 && row_ok && !s.full) {
          p.part_ml[(rec * p.R + r) * 2 + 0] = -INFINITY;
          p.part_ml[(rec * p.R + r) * 2 + 1] = 0.f;
        }
        continue;
      }
      int wi = 0;
      for (int t = s.t0; t < s.t1; ++t) {
        if (!attn_tile_live(p, s, t)) continue;
        const bool first = (wi == 0), last = (wi == nwork - 1);
        const int buf = n % kPairSP;
        const uint32_t sp = tmem + lane_off + 128 + 128 * buf;   // SP[buf] of this lane quarter
        mbar_wait(&s_full[buf], (n / kPairSP) & 1, ERR_WAIT_MMA);
        tc_fence_after();
        float x[64];
        {
          float (&x0)[32] = *reinterpret_cast<float (*)[32]>(&x[0]);
          float (&x1)[32] = *reinterpret_cast<float (*)[32]>(&x[32]);
          tmem_ld32(sp + kh * 64, x0);
          tmem_ld32(sp + kh * 64 + 32, x1);
        }
        tmem_ld_wait();
        const int nvalid = (t < p.n_ctx_tiles) ? min(kKeyTile, s.L - t * kKeyTile) : p.S;
        if (nvalid < kKeyTile) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (kh * 64 + j >= nvalid) x[j] = -INFINITY;
        }
        // row maximum of the raw scores, then the partner's half; scaling by
        // log2(e)/sqrt(D) > 0 commutes with the maximum
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = fmax3(x[k], x[k + 8], x[k + 16]);
#pragma unroll
        for (int j = 24; j + 16 <= 64; j += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], x[j + k], x[j + 8 + k]);
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], x[56 + k]);
        const float pmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                 fmaxf(mx[6], mx[7]));
        // the exchange also tells each warp that its partner has read its S: P may now be
        // written over the first 64 columns of SP[buf]
        float* xm = xch + (n & 1) * 256;
        xm[kh * 128 + r] = pmax;
        tc_fence_before();
        pair_sync(bar_id);
        tc_fence_after();
        const float omax = xm[(1 - kh) * 128 + r];
        const float tmax = fmaxf(pmax, omax) * sc;
        if (first) {
          m_run = tmax;
          l_run = 0.f;
        } else if (tmax > m_run + 8.0f) {
          const float alpha = ex2_approx(m_run - tmax);
          m_run = tmax;
          l_run *= alpha;
          // every PV so far (the last one used SP[(n-1) % 3]) must be done before O is touched
          pair_rescale(tmem, lane_off, kh, alpha, &o_done[(n - 1) % kPairSP],
                       ((n - 1) / kPairSP) & 1);
        }
        // P = 2^(x*scale - m) rounded to bf16, two per TMEM column (keys 64kh.. -> columns
        // 32kh.. of SP[buf]); the running sum adds the fp32 values
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
          tmem_st16(sp + kh * 32 + 16 * k, pk);
          if constexpr (kSplitP) tmem_st16(sp + 64 + kh * 32 + 16 * k, pl);
        }
        l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        tmem_st_wait();
        tc_fence_before();
        hand_off(&p_full[buf]);
        if (last)
          pair_epilogue(p.out, p.part_o, p.part_ml, p.lse, p.S, p.Hq,
                        p.R, tmem, lane_off, kh, r, row_ok, xch, bar_id, &o_done[buf],
                        (n / kPairSP) & 1, o_free, even, lane, m_run, l_run, s.full, s.b, s_tok,
                        head, rec);
        ++n;
        ++wi;
      }
    }
  }

  // No CTA of the pair leaves (or frees its TMEM) while the other may still signal its
  // barriers or while pair MMAs may still write its TMEM.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == kQkWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace td
