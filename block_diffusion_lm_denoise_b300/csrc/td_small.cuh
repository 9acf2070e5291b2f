// td_small.cuh -- the bandwidth-trivial steps of the denoise step:
//   embed_kernel          h0[r] = bf16(emb[tokens[r]] + pos[r % S])
//   adaln_slab_kernel     x_mod = bf16(LN(h) * (1 + scale) + shift), m = E + phi; also writes
//                         the gate row m[2] for the gated-residual epilogue
//   merge_commit_kernel   merges the LM head's per-tile (max, argmax, exp-sum) partials into
//                         conf / pred and applies the confidence-masking commit rule
//                         ("NVIDIA、Nemotron-Labs-TwoTowerを公開…", news.chathome.org,
//                         generation and evaluation paragraphs)
#pragma once

#include "td_ptx.cuh"

namespace td {

// One CTA per row; 8 bf16 per thread per step.
__global__ void embed_kernel(const int* __restrict__ tokens, const uint16_t* __restrict__ emb,
                             const uint16_t* __restrict__ pos, uint16_t* __restrict__ h, int S,
                             int d, int V, const int* skip) {
  if (skip != nullptr && *skip != 0) return;
  const int r = blockIdx.x;
  int tok = tokens[r];
  if (tok < 0 || tok > V) {     // not a vocabulary id nor [MASK]: flag it, read [MASK]
    if (threadIdx.x == 0) record_error(ERR_BAD_TOKEN);
    tok = V;
  }
  const uint4* e = reinterpret_cast<const uint4*>(emb + (size_t)tok * d);
  const uint4* q = reinterpret_cast<const uint4*>(pos + (size_t)(r % S) * d);
  uint4* o = reinterpret_cast<uint4*>(h + (size_t)r * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) {
    const uint4 a = __ldg(&e[i]);
    const uint4 b = __ldg(&q[i]);
    uint4 w;
    w.x = pack_bf16x2(bf16lo_to_f32(a.x) + bf16lo_to_f32(b.x), bf16hi_to_f32(a.x) + bf16hi_to_f32(b.x));
    w.y = pack_bf16x2(bf16lo_to_f32(a.y) + bf16lo_to_f32(b.y), bf16hi_to_f32(a.y) + bf16hi_to_f32(b.y));
    w.z = pack_bf16x2(bf16lo_to_f32(a.z) + bf16lo_to_f32(b.z), bf16hi_to_f32(a.z) + bf16hi_to_f32(b.z));
    w.w = pack_bf16x2(bf16lo_to_f32(a.w) + bf16lo_to_f32(b.w), bf16hi_to_f32(a.w) + bf16hi_to_f32(b.w));
    o[i] = w;
  }
}

constexpr int kAdaMaxD = 8192;

// Column-slab layout: a CTA of d / 8 threads owns kAdaSlabRows rows; thread t owns columns
// 8t .. 8t + 7 of every one of them and loads its eight-element slice of each row, all loads
// in flight together. Row statistics in fp32: each thread takes the mean and the sum of
// squared deviations of its own eight values (two passes over registers), and these pairs
// are merged across the warp and then across the CTA with the pairwise update of Chan, Golub
// and LeVeque ("Updating formulae and a pairwise algorithm for computing sample variances",
// 1979): for parts of sizes na, nb with means ma, mb and squared-deviation sums Qa, Qb,
// mean = ma + (mb - ma) nb / n and Q = Qa + Qb + (mb - ma)^2 na nb / n, n = na + nb. One
// CTA-wide exchange instead of one for the mean and one for the variance. The modulation
// values (1 + scale, shift) for the thread's columns are loaded while that exchange runs.
constexpr int kAdaSlabRows = 4;

__device__ __forceinline__ void chan_merge(float& n, float& m, float& q, float nb, float mb,
                                           float qb) {
  const float nn = n + nb;
  if (nn > 0.f) {
    const float dm = mb - m;
    const float w = nb / nn;
    m += dm * w;
    q += qb + dm * dm * n * w;
  }
  n = nn;
}

__global__ void __launch_bounds__(1024)
    adaln_slab_kernel(const uint16_t* __restrict__ h, const float* __restrict__ E,
                      const float* __restrict__ phi, int rows, int d, float eps,
                      uint16_t* __restrict__ x_mod, float* __restrict__ gate_out,
                      const int* skip) {
  constexpr int R = kAdaSlabRows;
  __shared__ float2 red[R][32];         // [row][warp] (mean, squared-deviation sum)
  __shared__ float2 stat[R];            // per row (mean, rstd)
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const int nwarps = blockDim.x >> 5;
  const int c0 = 8 * t;
  const int r0 = blockIdx.x * R;
  const bool skipped = skip != nullptr && *skip != 0;
  uint4 raw[R];
#pragma unroll
  for (int i = 0; i < R; ++i)
    raw[i] = (r0 + i < rows) ? *reinterpret_cast<const uint4*>(h + (size_t)(r0 + i) * d + c0)
                             : make_uint4(0, 0, 0, 0);
  if (skipped) return;
  if (gate_out != nullptr && blockIdx.x == 0) {
    const float4* e2 = reinterpret_cast<const float4*>(E + 2 * d + c0);
    const float4* p2 = reinterpret_cast<const float4*>(phi + 2 * d + c0);
    const float4 a0 = __ldg(&e2[0]), a1 = __ldg(&e2[1]), b0 = __ldg(&p2[0]), b1 = __ldg(&p2[1]);
    float4* g = reinterpret_cast<float4*>(gate_out + c0);
    g[0] = make_float4(a0.x + b0.x, a0.y + b0.y, a0.z + b0.z, a0.w + b0.w);
    g[1] = make_float4(a1.x + b1.x, a1.y + b1.y, a1.z + b1.z, a1.w + b1.w);
  }
  auto unpack = [](const uint4& w, float (&x)[8]) {
    x[0] = bf16lo_to_f32(w.x); x[1] = bf16hi_to_f32(w.x);
    x[2] = bf16lo_to_f32(w.y); x[3] = bf16hi_to_f32(w.y);
    x[4] = bf16lo_to_f32(w.z); x[5] = bf16hi_to_f32(w.z);
    x[6] = bf16lo_to_f32(w.w); x[7] = bf16hi_to_f32(w.w);
  };
  // per-thread statistics of its eight values, then merged over the warp; the xor partners
  // hold equal counts, so the merge reduces to mean = (ma + mb) / 2, Q = Qa + Qb + dm^2 n / 2
  float mu[R], q[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    float x[8];
    unpack(raw[i], x);
    const float m = (((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]))) * 0.125f;
    float qq = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float a = x[j] - m;
      qq += a * a;
    }
    mu[i] = m;
    q[i] = qq;
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float half_n = 4.0f * (float)o;   // n / 2 with n = 8 o values on each side
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const float mb = __shfl_xor_sync(0xffffffffu, mu[i], o);
      const float qb = __shfl_xor_sync(0xffffffffu, q[i], o);
      const float dm = mb - mu[i];
      mu[i] = 0.5f * (mu[i] + mb);
      q[i] = (q[i] + qb) + dm * dm * half_n;
    }
  }
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < R; ++i) red[i][warp] = make_float2(mu[i], q[i]);
  // modulation slice: shift = E[0] + phi[0], 1 + scale = 1 + E[1] + phi[1]
  float sh[8], sc[8];
  {
    const float4* e0 = reinterpret_cast<const float4*>(E + c0);
    const float4* e1 = reinterpret_cast<const float4*>(E + d + c0);
    const float4* p0 = reinterpret_cast<const float4*>(phi + c0);
    const float4* p1 = reinterpret_cast<const float4*>(phi + d + c0);
    const float4 a0 = __ldg(&e0[0]), a1 = __ldg(&e0[1]), b0 = __ldg(&p0[0]), b1 = __ldg(&p0[1]);
    const float4 c0v = __ldg(&e1[0]), c1v = __ldg(&e1[1]), d0 = __ldg(&p1[0]), d1 = __ldg(&p1[1]);
    sh[0] = a0.x + b0.x; sh[1] = a0.y + b0.y; sh[2] = a0.z + b0.z; sh[3] = a0.w + b0.w;
    sh[4] = a1.x + b1.x; sh[5] = a1.y + b1.y; sh[6] = a1.z + b1.z; sh[7] = a1.w + b1.w;
    sc[0] = 1.0f + (c0v.x + d0.x); sc[1] = 1.0f + (c0v.y + d0.y);
    sc[2] = 1.0f + (c0v.z + d0.z); sc[3] = 1.0f + (c0v.w + d0.w);
    sc[4] = 1.0f + (c1v.x + d1.x); sc[5] = 1.0f + (c1v.y + d1.y);
    sc[6] = 1.0f + (c1v.z + d1.z); sc[7] = 1.0f + (c1v.w + d1.w);
  }
  __syncthreads();
  for (int i = warp; i < R; i += nwarps) {   // row i merged over the CTA's warps (256 values each)
    float n = 0.f, m = 0.f, qq = 0.f;
    if (lane < nwarps) {
      const float2 v = red[i][lane];
      n = 256.f;
      m = v.x;
      qq = v.y;
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float nb = __shfl_xor_sync(0xffffffffu, n, o);
      const float mb = __shfl_xor_sync(0xffffffffu, m, o);
      const float qb = __shfl_xor_sync(0xffffffffu, qq, o);
      chan_merge(n, m, qq, nb, mb, qb);
    }
    if (lane == 0) stat[i] = make_float2(m, 1.0f / sqrtf(qq / (float)d + eps));
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < R; ++i) {
    if (r0 + i >= rows) break;
    const float2 st = stat[i];
    float x[8];
    unpack(raw[i], x);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = pack_bf16x2((x[2 * j] - st.x) * st.y * sc[2 * j] + sh[2 * j],
                         (x[2 * j + 1] - st.x) * st.y * sc[2 * j + 1] + sh[2 * j + 1]);
    *reinterpret_cast<uint4*>(x_mod + (size_t)(r0 + i) * d + c0) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Any d that is a multiple of 8 (or E / phi off a 16-byte boundary): one CTA per row,
// scalar loads.
__global__ void __launch_bounds__(256)
    adaln_modulate_generic_kernel(const uint16_t* __restrict__ h, const float* __restrict__ E,
                                  const float* __restrict__ phi, int d, float eps,
                                  uint16_t* __restrict__ x_mod, float* __restrict__ gate_out,
                                  const int* skip) {
  if (skip != nullptr && *skip != 0) return;
  __shared__ float red[8];
  const int r = blockIdx.x;
  const uint16_t* hr = h + (size_t)r * d;
  float s = 0.f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) s += __uint_as_float((uint32_t)hr[c] << 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
  const float mean = t / (float)d;
  __syncthreads();
  float ss = 0.f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    const float a = __uint_as_float((uint32_t)hr[c] << 16) - mean;
    ss += a * a;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  t = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
  const float rstd = 1.0f / sqrtf(t / (float)d + eps);
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    const float x = __uint_as_float((uint32_t)hr[c] << 16);
    const float y = (x - mean) * rstd * (1.0f + (E[d + c] + phi[d + c])) + (E[c] + phi[c]);
    x_mod[(size_t)r * d + c] = (uint16_t)(pack_bf16x2(y, 0.f) & 0xFFFFu);
  }
  if (gate_out != nullptr && r == 0)
    for (int c = threadIdx.x; c < d; c += blockDim.x) gate_out[c] = E[2 * d + c] + phi[2 * d + c];
}

// Rows the LM head evaluates in a denoise step: those still masked when the step starts
// (committed rows need no logits); under the left-to-right rule before the last step, only
// the lowest masked row of each sequence (the only one that can commit). One CTA of
// kRowsThreads threads; thread t owns the contiguous rows [t * per, (t + 1) * per).
// row_pos[r] = index of row r among the selected rows (row order kept), or -1;
// *count = number of selected rows.
constexpr int kRowsThreads = 1024;
constexpr int kRuleConfidence = 0;
constexpr int kRuleLeftToRight = 1;

__device__ __forceinline__ bool lm_row_selected(const unsigned char* masked, int r, int S,
                                                bool first_only) {
  if (masked[r] == 0) return false;
  if (!first_only) return true;
  for (int j = r - r % S; j < r; ++j)
    if (masked[j] != 0) return false;
  return true;
}

__global__ void __launch_bounds__(kRowsThreads)
    lm_rows_kernel(const unsigned char* __restrict__ masked, int M, int S, int first_only,
                   int* __restrict__ row_pos, int* __restrict__ count, const int* skip) {
  if (skip != nullptr && *skip != 0) return;
  __shared__ int warp_tot[kRowsThreads / 32];
  const int per = (M + kRowsThreads - 1) / kRowsThreads;
  const int r0 = min(M, (int)threadIdx.x * per), r1 = min(M, r0 + per);
  int n = 0;
  for (int r = r0; r < r1; ++r) n += lm_row_selected(masked, r, S, first_only != 0);
  // exclusive scan of n over the block: within the warp, then over the warp totals
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_tot[lane] = w;   // inclusive over warps
  }
  __syncthreads();
  int base = incl - n + (warp > 0 ? warp_tot[warp - 1] : 0);
  for (int r = r0; r < r1; ++r)
    row_pos[r] = lm_row_selected(masked, r, S, first_only != 0) ? base++ : -1;
  if (threadIdx.x == kRowsThreads - 1) *count = warp_tot[31];
}

// Copies row r of h to row row_pos[r] of h_out when row_pos[r] >= 0 (a step without layers:
// the caller's hidden states go to the LM head as they are). One CTA per row.
__global__ void gather_rows_kernel(const uint16_t* __restrict__ h, const int* __restrict__ row_pos,
                                   uint16_t* __restrict__ h_out, int d, const int* skip) {
  if (skip != nullptr && *skip != 0) return;
  const int r = blockIdx.x;
  const int rp = row_pos[r];
  if (rp < 0) return;
  const uint4* src = reinterpret_cast<const uint4*>(h + (size_t)r * d);
  uint4* dst = reinterpret_cast<uint4*>(h_out + (size_t)rp * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) dst[i] = src[i];
}

// One CTA per sequence, one warp per position (up to 32 warps, looping beyond): a warp merges
// the row's vocabulary-slice partials (max, lowest argmax, exp-sum), lowest slice first so
// the lowest id wins ties; then warp 0 applies the commit rule to the sequence.
__global__ void __launch_bounds__(1024)
    merge_commit_kernel(const float* __restrict__ part_max, const int* __restrict__ part_arg,
                        const float* __restrict__ part_sum, int n_tiles, int S, float gamma,
                        int force_all, int rule, int* tokens, unsigned char* masked,
                        float* conf_out,
                        int* pred_out, int* n_committed, int* all_done, int* counters,
                        const int* skip, int* steps_taken, const int* row_pos,
                        cudaGraphConditionalHandle next_step, int set_next_step) {
  // skip: the decode loop already finished; steps_taken (optional) counts the steps that ran;
  // row_pos (optional): the partials hold only the rows masked at the step start, row r at
  // row_pos[r]; the other rows were not evaluated and get conf 0, pred -1; with set_next_step
  // (inside a decode-loop graph) the condition of the next step's node is set to "positions
  // left"
  if (skip != nullptr && *skip != 0) return;
  if (steps_taken != nullptr && blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(steps_taken, 1);
  __shared__ float s_conf[64];
  __shared__ int s_pred[64];
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  for (int i = warp; i < S; i += nwarps) {
    const size_t row = (size_t)b * S + i;
    size_t prow = row;
    if (row_pos != nullptr) {
      const int rp = row_pos[row];
      if (rp < 0) {
        if (lane == 0) {
          s_conf[i] = 0.f;
          s_pred[i] = -1;
          conf_out[row] = 0.f;
          pred_out[row] = -1;
        }
        continue;
      }
      prow = (size_t)rp;
    }
    const float* pm = part_max + prow * n_tiles;
    const int* pa = part_arg + prow * n_tiles;
    const float* ps = part_sum + prow * n_tiles;
    // lane-local pass over slices lane, lane+32, ..., eight at a time (the loads of a batch
    // are independent): max with the lowest slice on ties, and the exp-sum relative to a
    // running max (rescaled when it grows)
    float m = -INFINITY, sum = 0.f;
    int mt = 0x7fffffff;
    for (int t0 = lane; t0 < n_tiles; t0 += 32 * 8) {
      float vm[8], vs[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int t = t0 + 32 * j;
        vm[j] = t < n_tiles ? __ldg(&pm[t]) : -INFINITY;
        vs[j] = t < n_tiles ? __ldg(&ps[t]) : 0.f;
      }
      float cm = vm[0];
      int ct = t0;
#pragma unroll
      for (int j = 1; j < 8; ++j)
        if (vm[j] > cm) {
          cm = vm[j];
          ct = t0 + 32 * j;
        }
      if (cm > m) {
        sum = (m == -INFINITY) ? 0.f : sum * ex2_approx((m - cm) * 1.4426950408889634f);
        m = cm;
        mt = ct;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (vm[j] != -INFINITY) sum += vs[j] * ex2_approx((vm[j] - m) * 1.4426950408889634f);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const int t2 = __shfl_xor_sync(0xffffffffu, mt, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, sum, o);
      const float mm = fmaxf(m, m2);
      const float a = (m == -INFINITY) ? 0.f : sum * ex2_approx((m - mm) * 1.4426950408889634f);
      const float c = (m2 == -INFINITY) ? 0.f : s2 * ex2_approx((m2 - mm) * 1.4426950408889634f);
      if (m2 > m || (m2 == m && t2 < mt)) mt = t2;
      m = mm;
      sum = a + c;
    }
    if (lane == 0) {
      const float c = 1.0f / sum;
      const int pr = pa[mt];
      s_conf[i] = c;
      s_pred[i] = pr;
      conf_out[row] = c;
      pred_out[row] = pr;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // positions lane and lane + 32 (S <= 64)
    int n_commit = 0, remaining = 0;
    bool msk[2], thr[2];
    float cf[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      msk[k] = (i < S) && masked[(size_t)b * S + i] != 0;
      cf[k] = (i < S) ? s_conf[i] : -INFINITY;
      thr[k] = msk[k] && cf[k] >= gamma;
    }
    const unsigned any_thr = __ballot_sync(0xffffffffu, thr[0] || thr[1]);
    const unsigned any_msk = __ballot_sync(0xffffffffu, msk[0] || msk[1]);
    bool take[2] = {false, false};
    if (force_all) {
      take[0] = msk[0]; take[1] = msk[1];
    } else if (rule == kRuleLeftToRight) {
      // the lowest-index masked position, whatever its confidence
      const unsigned m0 = __ballot_sync(0xffffffffu, msk[0]);
      const unsigned m1 = __ballot_sync(0xffffffffu, msk[1]);
      const int lo = m0 ? __ffs(m0) - 1 : (m1 ? 32 + __ffs(m1) - 1 : -1);
      take[0] = (lane == lo);
      take[1] = (lane + 32 == lo);
    } else if (any_thr) {
      take[0] = thr[0]; take[1] = thr[1];
    } else if (any_msk) {
      // the most confident masked position, lowest index on ties
      float best = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = lane + 32 * k;
        if (msk[k] && (cf[k] > best || (cf[k] == best && i < bi))) { best = cf[k]; bi = i; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        if (b2 > best || (b2 == best && i2 < bi)) { best = b2; bi = i2; }
      }
      take[0] = (lane == bi);
      take[1] = (lane + 32 == bi);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      if (take[k]) {
        tokens[(size_t)b * S + i] = s_pred[i];
        masked[(size_t)b * S + i] = 0;
        ++n_commit;
      } else if (msk[k]) {
        ++remaining;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n_commit += __shfl_xor_sync(0xffffffffu, n_commit, o);
      remaining += __shfl_xor_sync(0xffffffffu, remaining, o);
    }
    if (lane == 0) {
      n_committed[b] = n_commit;
      // counters[0]: masked positions left over all sequences; counters[1]: CTAs finished.
      if (remaining) atomicAdd(&counters[0], remaining);
      __threadfence();
      const int ticket = atomicAdd(&counters[1], 1);
      if (ticket == (int)gridDim.x - 1) {
        __threadfence();
        const int left = atomicAdd(&counters[0], 0);
        *all_done = (left == 0) ? 1 : 0;
        if (set_next_step) cudaGraphSetConditional(next_step, left != 0 ? 1u : 0u);
        counters[0] = 0;
        counters[1] = 0;
      }
    }
  }
}

// Rotary table of a step: row r = b*S + i sits at position ctx_len[b] + i (Lmax without
// ctx_len); pair j of a head turns by pos * theta^(-2j / head_dim). The angle and its cosine
// and sine are taken in double precision, then stored as float.
__global__ void rope_table_kernel(const int* __restrict__ ctx_len, int B, int S, int Lmax,
                                  int head_dim, double theta, float2* __restrict__ cs,
                                  const int* skip) {
  if (skip != nullptr && *skip != 0) return;
  const int half = head_dim / 2;
  const int total = B * S * half;
  for (int x = blockIdx.x * blockDim.x + threadIdx.x; x < total; x += gridDim.x * blockDim.x) {
    const int j = x % half;
    const int r = x / half;
    const int b = r / S, i = r % S;
    const int L = ctx_len != nullptr ? ctx_len[b] : Lmax;
    const double ang = (double)(L + i) * pow(theta, -2.0 * (double)j / (double)head_dim);
    double sn, cn;
    sincos(ang, &sn, &cn);
    cs[x] = make_float2((float)cn, (float)sn);
  }
}

// adaLN-single timestep map: phi(t) = W_t e(t / T) + b_t for t = 1..T, e the 256-wide
// sinusoidal embedding of s = 1000 t / T (e[j] = cos(s w_j), e[128 + j] = sin(s w_j),
// w_j = 10000^(-j / 128)). One warp per output row k of W_t [6d, 256] (its 256 weights, eight
// a lane, read once) for a chunk of up to kTsChunk steps; the embeddings of the chunk are
// built in shared memory, everything in double precision, the result rounded to float once.
constexpr int kTsDim = 256;
constexpr int kTsChunk = 16;
constexpr int kTsWarps = 8;

__global__ void __launch_bounds__(32 * kTsWarps)
    timestep_table_kernel(const float* __restrict__ w_t, const float* __restrict__ b_t,
                          int rows, int T, float* __restrict__ phi) {
  __shared__ double emb[kTsChunk][kTsDim];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = blockIdx.x * kTsWarps + warp;
  double w[kTsDim / 32];
  if (k < rows) {
#pragma unroll
    for (int i = 0; i < kTsDim / 32; ++i) w[i] = (double)__ldg(&w_t[(size_t)k * kTsDim + lane + 32 * i]);
  }
  const double bias = k < rows ? (double)__ldg(&b_t[k]) : 0.0;
  for (int t0 = 0; t0 < T; t0 += kTsChunk) {
    const int nt = min(kTsChunk, T - t0);
    __syncthreads();
    for (int x = threadIdx.x; x < nt * (kTsDim / 2); x += blockDim.x) {
      const int tt = x / (kTsDim / 2), j = x % (kTsDim / 2);
      const double s = 1000.0 * (double)(t0 + tt + 1) / (double)T;
      const double a = s * pow(10000.0, -(double)j / (double)(kTsDim / 2));
      double sn, cn;
      sincos(a, &sn, &cn);
      emb[tt][j] = cn;
      emb[tt][kTsDim / 2 + j] = sn;
    }
    __syncthreads();
    if (k >= rows) continue;
    for (int tt = 0; tt < nt; ++tt) {
      double acc = 0.0;
#pragma unroll
      for (int i = 0; i < kTsDim / 32; ++i) acc = fma(w[i], emb[tt][lane + 32 * i], acc);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) phi[(size_t)(t0 + tt) * rows + k] = (float)(acc + bias);
    }
  }
}

// One thread waits, through the same bounded wait every kernel uses, on a barrier that
// nothing completes: the wait must give up after limit_ns and record ERR_WAIT_EPI.
__global__ void wait_check_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_wait(&bar, 0, ERR_WAIT_EPI, limit_ns);
}

// Context-cache append: row ctx_len[b] + i of KV head g of a layer's cache receives
// token i of head g of the block's keys / values ([B, S, Hkv, D], token-major). One thread
// per 16-byte chunk; sequences whose cache would pass Lmax are skipped (flagged by the
// length update below).
// With page_table set, the caches are pools [n_pages][Hkv][128][D] and position pos of
// sequence b lives in page page_table[b * max_pages + pos / 128], row pos % 128. A sequence
// any of whose new positions maps to an entry outside [0, n_pages) is skipped whole (the
// length update flags it and keeps its length).

// True if every page-table entry of positions L .. L + S - 1 of sequence b is in range
// (S <= 64 < 128: the positions span at most two pages).
__device__ __forceinline__ bool append_pages_ok(const int* page_table, int max_pages,
                                                int n_pages, int b, int L, int S) {
  const int p0 = page_table[(size_t)b * max_pages + L / 128];
  const int p1 = page_table[(size_t)b * max_pages + (L + S - 1) / 128];
  return p0 >= 0 && p0 < n_pages && p1 >= 0 && p1 < n_pages;
}

__global__ void kv_append_kernel(const uint16_t* __restrict__ k_new,
                                 const uint16_t* __restrict__ v_new, uint16_t* __restrict__ k_ctx,
                                 uint16_t* __restrict__ v_ctx, const int* __restrict__ ctx_len,
                                 int B, int S, int Hkv, int D, int Lmax,
                                 const int* __restrict__ page_table, int max_pages, int n_pages) {
  const int c16 = D / 8;
  const long long total = (long long)B * S * Hkv * c16;
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < total;
       x += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(x % c16);
    long long row = x / c16;               // (b, i, g) of the block tensor
    const int g = (int)(row % Hkv);
    const int i = (int)((row / Hkv) % S);
    const int b = (int)(row / ((long long)Hkv * S));
    const int L = ctx_len[b];
    if (L < 0 || L + S > Lmax) continue;
    if (page_table != nullptr && !append_pages_ok(page_table, max_pages, n_pages, b, L, S))
      continue;
    const int pos = L + i;
    size_t dst;
    if (page_table != nullptr) {
      const int page = page_table[(size_t)b * max_pages + pos / 128];
      dst = (((size_t)page * Hkv + g) * 128 + (size_t)(pos % 128)) * D + (size_t)c * 8;
    } else {
      dst = (((size_t)b * Hkv + g) * Lmax + (size_t)pos) * D + (size_t)c * 8;
    }
    const size_t src = (size_t)row * D + (size_t)c * 8;
    *reinterpret_cast<uint4*>(k_ctx + dst) = *reinterpret_cast<const uint4*>(k_new + src);
    *reinterpret_cast<uint4*>(v_ctx + dst) = *reinterpret_cast<const uint4*>(v_new + src);
  }
}

// After every layer's append: ctx_len[b] += S, or the overflow (or, paged, an out-of-range
// page entry of the new positions) is recorded and the length kept.
__global__ void kv_len_update_kernel(int* ctx_len, int B, int S, int Lmax,
                                     const int* __restrict__ page_table, int max_pages,
                                     int n_pages) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int L = ctx_len[b];
  if (L < 0 || L + S > Lmax) record_error(ERR_CTX_FULL);
  else if (page_table != nullptr && !append_pages_ok(page_table, max_pages, n_pages, b, L, S))
    record_error(ERR_BAD_PAGE);
  else ctx_len[b] = L + S;
}

}  // namespace td
