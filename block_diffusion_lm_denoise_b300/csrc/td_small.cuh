// td_small.cuh -- the bandwidth-trivial steps of the denoise step:
//   embed_kernel          h0[r] = bf16(emb[tokens[r]] + pos[r % S])
//   adaln_modulate_kernel x_mod = bf16(LN(h) * (1 + scale) + shift), m = E + phi; also writes
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
                             int d, int V) {
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

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
  return t;
}

// One CTA (256 threads) per row; the row is held in registers (d <= 256 * 8 * kMaxVec).
constexpr int kAdaThreads = 256;
constexpr int kAdaMaxVec = 4;   // d <= 8192

__global__ void __launch_bounds__(kAdaThreads)
    adaln_modulate_kernel(const uint16_t* __restrict__ h, const float* __restrict__ E,
                          const float* __restrict__ phi, int d, float eps,
                          uint16_t* __restrict__ x_mod, float* __restrict__ gate_out) {
  __shared__ float red[kAdaThreads / 32];
  const int r = blockIdx.x;
  const uint4* hr = reinterpret_cast<const uint4*>(h + (size_t)r * d);
  const int nv = d / 8;
  float x[kAdaMaxVec][8];
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kAdaMaxVec; ++k) {
    const int i = threadIdx.x + k * kAdaThreads;
    if (i < nv) {
      const uint4 a = hr[i];
      x[k][0] = bf16lo_to_f32(a.x); x[k][1] = bf16hi_to_f32(a.x);
      x[k][2] = bf16lo_to_f32(a.y); x[k][3] = bf16hi_to_f32(a.y);
      x[k][4] = bf16lo_to_f32(a.z); x[k][5] = bf16hi_to_f32(a.z);
      x[k][6] = bf16lo_to_f32(a.w); x[k][7] = bf16hi_to_f32(a.w);
#pragma unroll
      for (int j = 0; j < 8; ++j) s += x[k][j];
    }
  }
  const float mean = block_sum(s, red) / (float)d;
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kAdaMaxVec; ++k) {
    const int i = threadIdx.x + k * kAdaThreads;
    if (i < nv) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float t = x[k][j] - mean;
        ss += t * t;
      }
    }
  }
  const float var = block_sum(ss, red) / (float)d;
  const float rstd = 1.0f / sqrtf(var + eps);
  uint4* out = reinterpret_cast<uint4*>(x_mod + (size_t)r * d);
#pragma unroll
  for (int k = 0; k < kAdaMaxVec; ++k) {
    const int i = threadIdx.x + k * kAdaThreads;
    if (i < nv) {
      float y[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = i * 8 + j;
        const float shift = E[c] + phi[c];
        const float scale = E[d + c] + phi[d + c];
        y[j] = (x[k][j] - mean) * rstd * (1.0f + scale) + shift;
      }
      out[i] = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                          pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
    }
  }
  if (gate_out != nullptr && r == 0) {
    for (int c = threadIdx.x; c < d; c += blockDim.x) gate_out[c] = E[2 * d + c] + phi[2 * d + c];
  }
}

// One CTA per sequence, 32*S2 threads (S2 = S rounded up to a warp multiple / 32 warps max):
// warp w merges rows w, w + nwarps, ... over the n_tiles vocabulary partials (increasing
// vocabulary order, so the lowest id wins ties), then warp 0 applies the commit rule.
constexpr int kCommitThreads = 256;

__global__ void __launch_bounds__(kCommitThreads)
    merge_commit_kernel(const float* __restrict__ part_max, const int* __restrict__ part_arg,
                        const float* __restrict__ part_sum, int n_tiles, int S, float gamma,
                        int force_all, int* tokens, unsigned char* masked, float* conf_out,
                        int* pred_out, int* n_committed, int* all_done, int* counters) {
  __shared__ float s_conf[64];
  __shared__ int s_pred[64];
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  for (int i = warp; i < S; i += nwarps) {
    const size_t row = (size_t)b * S + i;
    const float* pm = part_max + row * n_tiles;
    const int* pa = part_arg + row * n_tiles;
    const float* ps = part_sum + row * n_tiles;
    // lane-local pass: max with the lowest tile index on ties (tiles visited in order)
    float m = -INFINITY;
    int mt = 0x7fffffff;
    for (int t = lane; t < n_tiles; t += 32) {
      const float v = pm[t];
      if (v > m) { m = v; mt = t; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const int t2 = __shfl_xor_sync(0xffffffffu, mt, o);
      if (m2 > m || (m2 == m && t2 < mt)) { m = m2; mt = t2; }
    }
    float s = 0.f;
    for (int t = lane; t < n_tiles; t += 32) s += ps[t] * ex2_approx((pm[t] - m) * 1.4426950408889634f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
      const float c = 1.0f / s;
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
        counters[0] = 0;
        counters[1] = 0;
      }
    }
  }
}

}  // namespace td
