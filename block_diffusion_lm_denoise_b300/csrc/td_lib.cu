// td_lib.cu -- the C ABI of the denoise step: argument validation, workspace carving,
// TMA descriptor encoding, kernel selection and launch sequencing. Device code lives in the
// td_*.cuh headers included below (one translation unit, so the device error word is one
// symbol without relocatable device code).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "../../include/td.h"
#include "td_attention.cuh"
#include "td_attention_pair.cuh"
#include "td_gemm.cuh"
#include "td_ptx.cuh"
#include "td_small.cuh"

namespace {

using namespace td;

constexpr float kLnEps = 1e-6f;
constexpr size_t kAlign = 256;

size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

#define TD_CUDA(call)                                   \
  do {                                                  \
    cudaError_t e__ = (call);                           \
    if (e__ != cudaSuccess) return TD_ERR_CUDA;         \
  } while (0)

// ------------------------------------------------------------------------------------------
// Driver entry point for tensor-map encoding (resolved once; no link-time libcuda).
// ------------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 tensor map of rank `rank` (dims innermost first, strides in bytes for dims 1..rank-1),
// box `box`, 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bd[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bd[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gd, gs, bd, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

// Dynamic shared-memory opt-in, done once per (kernel, device) so that no attribute call is
// made while a decode loop is being captured into a CUDA graph.
cudaError_t set_smem_raw(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  int& have = done[std::make_pair(kernel, dev)];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return set_smem_raw(reinterpret_cast<const void*>(kernel), bytes);
}

// ------------------------------------------------------------------------------------------
// Validation
// ------------------------------------------------------------------------------------------
td_status check_dims(const td_dims* dm, bool need_model) {
  if (!dm) return TD_ERR_INVALID_ARG;
  if (dm->B <= 0 || dm->S <= 0 || dm->D <= 0 || dm->Hq <= 0 || dm->Hkv <= 0 || dm->Lmax < 0)
    return TD_ERR_INVALID_ARG;
  if (need_model && (dm->d <= 0 || dm->V <= 0 || dm->n_layers < 0)) return TD_ERR_INVALID_ARG;
  if (dm->D != 64 && dm->D != 128) return TD_ERR_UNSUPPORTED;
  if (dm->Hq % dm->Hkv != 0) return TD_ERR_UNSUPPORTED;
  if (dm->S > 64) return TD_ERR_UNSUPPORTED;
  if ((long long)dm->B * dm->S > 65536) return TD_ERR_UNSUPPORTED;
  if (need_model && (dm->d % 64 != 0 || dm->d > 8192 || dm->V % 8 != 0)) return TD_ERR_UNSUPPORTED;
  return TD_OK;
}

td_status check_lm_dims(const td_dims* dm) {
  if (!dm) return TD_ERR_INVALID_ARG;
  if (dm->B <= 0 || dm->S <= 0 || dm->d <= 0 || dm->V <= 0) return TD_ERR_INVALID_ARG;
  if (dm->S > 64 || (long long)dm->B * dm->S > 65536) return TD_ERR_UNSUPPORTED;
  if (dm->d % 64 != 0 || dm->V % 8 != 0) return TD_ERR_UNSUPPORTED;
  return TD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ------------------------------------------------------------------------------------------
// Attention plan
// ------------------------------------------------------------------------------------------
struct AttnPlan {
  int G, Gc, NC, R, n_ctx_tiles, T, n_units, n_teams, ncta, max_seg;
  bool pair;    // head_dim 128: two chunks per SM pair (attn_pair_kernel)
  int NCT;      // pair kernel: CTA pairs per team
  bool split;   // some unit is shared by two teams: partials + merge pass
  long long total;
  size_t part_o_bytes, part_ml_bytes;
};

// A team walks one key range for all row chunks of its units: NC CTAs (one per 128-row
// chunk) or, for head_dim 128, ceil(NC / 2) CTA pairs (one chunk per SM of a pair).
//  - at least as many units as teams: if the units split evenly over >= 85% of the possible
//    teams, each team takes whole units (no merge pass); otherwise the (unit, tile) space is
//    cut into one equal range per team (split-K) and the partials are merged;
//  - fewer units than teams: every unit is cut into k = teams / units equal key ranges, so
//    team boundaries fall on unit boundaries and the merge combines exactly k partials.
AttnPlan plan_attention(const td_dims* dm, int nsm) {
  AttnPlan a{};
  a.G = dm->Hq / dm->Hkv;
  a.Gc = 1;
  for (int c = a.G; c >= 1; --c)
    if (a.G % c == 0 && dm->S * c <= 128) { a.Gc = c; break; }
  a.NC = a.G / a.Gc;
  a.R = dm->S * a.Gc;
  a.pair = dm->D == 128 && a.NC >= 2;
  a.NCT = (a.NC + 1) / 2;
  a.n_ctx_tiles = (dm->Lmax + kKeyTile - 1) / kKeyTile;
  a.T = a.n_ctx_tiles + 1;
  a.n_units = dm->B * dm->Hkv;
  a.total = (long long)a.n_units * a.T;
  const int team_ctas = a.pair ? 2 * a.NCT : a.NC;
  const int max_teams = std::max(1, nsm / team_ctas);
  if (a.n_units >= max_teams) {
    const int per = (a.n_units + max_teams - 1) / max_teams;
    const int even = (a.n_units + per - 1) / per;
    if (a.n_units % per == 0 && even * 100 >= max_teams * 85) {
      a.n_teams = even;
      a.split = false;
    } else {
      a.n_teams = max_teams;
      a.split = true;
    }
  } else {
    const int k = std::max(1, std::min(max_teams / a.n_units, a.T));
    a.n_teams = a.n_units * k;
    a.split = k > 1;
  }
  a.ncta = a.n_teams * team_ctas;
  const long long tiles = (a.total + a.n_teams - 1) / a.n_teams;
  a.max_seg = (int)((tiles + a.T - 1) / a.T) + 1;
  // partial records: sized for the largest plan any problem up to this one can take (every
  // possible team splitting its range), so that the workspace never shrinks as B grows and a
  // buffer sized for one batch serves every smaller one
  const long long tiles_bound = (a.total + max_teams - 1) / max_teams;
  const size_t recs_bound =
      (size_t)max_teams * a.NC * (size_t)(((tiles_bound + a.T - 1) / a.T) + 1);
  const size_t recs = std::max((size_t)a.n_teams * a.NC * a.max_seg, recs_bound);
  a.part_o_bytes = align_up(recs * a.R * dm->D * sizeof(float));
  a.part_ml_bytes = align_up(recs * a.R * 2 * sizeof(float));
  return a;
}

size_t attn_ws_bytes(const td_dims* dm, int nsm) {
  const AttnPlan a = plan_attention(dm, nsm);
  return a.part_o_bytes + a.part_ml_bytes;
}

// ------------------------------------------------------------------------------------------
// LM head plan
// ------------------------------------------------------------------------------------------
int lm_bn(int M) { return M <= 128 ? 128 : 256; }

size_t lm_ws_bytes(int M, int V) {
  const int nt = (V + lm_bn(M) - 1) / lm_bn(M);
  const size_t part = (size_t)M * nt;
  return align_up(part * 4) * 3 + kAlign;   // max, arg, sum, counters
}

// ------------------------------------------------------------------------------------------
// Launch helpers
// ------------------------------------------------------------------------------------------
template <int BN, int STAGES, int EPI>
td_status launch_gemm(const void* A, const void* Bm, int M, int N, int K, GemmParams gp,
                      cudaStream_t st, int nsm) {
  using L = GemmSmem<BN, STAGES>;
  CUtensorMap ma, mb;
  const uint64_t da[2] = {(uint64_t)K, (uint64_t)M}, sa[1] = {(uint64_t)K * 2};
  const uint32_t ba[2] = {64, 128};
  const uint64_t db[2] = {(uint64_t)K, (uint64_t)N}, sb[1] = {(uint64_t)K * 2};
  const uint32_t bb[2] = {64, (uint32_t)BN};
  if (!make_map(&ma, A, 2, da, sa, ba) || !make_map(&mb, Bm, 2, db, sb, bb)) return TD_ERR_CUDA;
  gp.M = M;
  gp.N = N;
  gp.K = K;
  gp.m_tiles = (M + 127) / 128;
  gp.n_tiles = (N + BN - 1) / BN;
  gp.items = gp.m_tiles * gp.n_tiles;
  auto kern = gemm_tn_kernel<BN, STAGES, EPI>;
  TD_CUDA(set_smem(kern, L::kBytes));
  const int grid = std::min(gp.items, nsm);
  kern<<<grid, 256, L::kBytes, st>>>(ma, mb, gp);
  TD_CUDA(cudaGetLastError());
  return TD_OK;
}

// 256 x 256 tiles on SM pairs: grid = two CTAs per pair tile, at most one pair per TPC.
template <int STAGES, int EPI>
td_status launch_gemm_pair(const void* A, const void* Bm, int M, int N, int K, GemmParams gp,
                           cudaStream_t st, int nsm) {
  using L = GemmPairSmem<STAGES, EPI>;
  CUtensorMap ma, mb;
  const uint64_t da[2] = {(uint64_t)K, (uint64_t)M}, sa[1] = {(uint64_t)K * 2};
  const uint64_t db[2] = {(uint64_t)K, (uint64_t)N}, sb[1] = {(uint64_t)K * 2};
  const uint32_t box[2] = {64, 128};
  if (!make_map(&ma, A, 2, da, sa, box) || !make_map(&mb, Bm, 2, db, sb, box)) return TD_ERR_CUDA;
  gp.M = M;
  gp.N = N;
  gp.K = K;
  gp.m_tiles = (M + 255) / 256;
  gp.n_tiles = (N + 255) / 256;
  gp.items = gp.m_tiles * gp.n_tiles;
  auto kern = gemm_pair_kernel<STAGES, EPI>;
  TD_CUDA(set_smem(kern, L::kBytes));
  const int grid = 2 * std::min(gp.items, std::max(1, nsm / 2));
  kern<<<grid, 256, L::kBytes, st>>>(ma, mb, gp);
  TD_CUDA(cudaGetLastError());
  return TD_OK;
}

// bn = 128: single-CTA 128 x 128 tiles (few rows); bn = 256: 256 x 256 tiles on SM pairs.
template <int EPI>
td_status gemm_dispatch(const void* A, const void* Bm, int M, int N, int K, GemmParams gp,
                        cudaStream_t st, int nsm, int bn) {
  if (bn == 128) return launch_gemm<128, 6, EPI>(A, Bm, M, N, K, gp, st, nsm);
  return launch_gemm_pair<pair_gemm_stages(EPI), EPI>(A, Bm, M, N, K, gp, st, nsm);
}

// adaLN-single modulation: the column-slab path for d = 256 * k (d <= 8192) with 16-byte
// aligned E and phi, else generic.
td_status launch_adaln(const void* h, const float* E, const float* phi, int rows, int d,
                       float eps, void* x_mod, float* gate, cudaStream_t st,
                       const int* skip = nullptr) {
  if (d % 256 == 0 && d / 8 <= 1024 && aligned16(E) && aligned16(phi)) {
    adaln_slab_kernel<<<(rows + kAdaSlabRows - 1) / kAdaSlabRows, d / 8, 0, st>>>(
        static_cast<const uint16_t*>(h), E, phi, rows, d, eps, static_cast<uint16_t*>(x_mod),
        gate, skip);
    TD_CUDA(cudaGetLastError());
    return TD_OK;
  }
  adaln_modulate_generic_kernel<<<rows, 256, 0, st>>>(static_cast<const uint16_t*>(h), E, phi,
                                                      d, eps, static_cast<uint16_t*>(x_mod),
                                                      gate, skip);
  TD_CUDA(cudaGetLastError());
  return TD_OK;
}

// Inside a decode-loop graph built from conditional nodes: the handle of the next step's node,
// which the commit kernel sets to "positions left".
struct NextStep {
  cudaGraphConditionalHandle handle = 0;
  int set = 0;
};

// With row_pos / m_count set, h holds only the rows masked at the step start (compacted,
// *m_count of them on the device) and the other rows are reported as not evaluated.
td_status run_lmhead_commit(const td_dims* dm, const void* h, const void* w_lm, float gamma,
                            int rule, int force_all, int* tokens, unsigned char* masked,
                            float* conf,
                            int* pred, int* n_committed, int* all_done, void* ws,
                            cudaStream_t st, int nsm, const int* skip = nullptr,
                            int* steps = nullptr, const int* row_pos = nullptr,
                            const int* m_count = nullptr,
                            const NextStep& next = NextStep{}) {
  const int M = dm->B * dm->S;
  const int V = dm->V;
  const int bn = lm_bn(M);
  const int nt = (V + bn - 1) / bn;
  const size_t part = (size_t)M * nt;
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* pmax = reinterpret_cast<float*>(w);
  int* parg = reinterpret_cast<int*>(w + align_up(part * 4));
  float* psum = reinterpret_cast<float*>(w + 2 * align_up(part * 4));
  int* counters = reinterpret_cast<int*>(w + 3 * align_up(part * 4));
  GemmParams gp{};
  gp.part_max = pmax;
  gp.part_arg = parg;
  gp.part_sum = psum;
  gp.skip = skip;
  gp.m_count = m_count;
  td_status s = gemm_dispatch<EPI_LMHEAD>(h, w_lm, M, V, dm->d, gp, st, nsm, bn);
  if (s != TD_OK) return s;
  TD_CUDA(cudaMemsetAsync(counters, 0, 2 * sizeof(int), st));
  merge_commit_kernel<<<dm->B, 32 * std::min(dm->S, 32), 0, st>>>(pmax, parg, psum, nt, dm->S, gamma,
                                                         force_all, rule, tokens, masked, conf,
                                                         pred,
                                                         n_committed, all_done, counters,
                                                         skip, steps, row_pos, next.handle,
                                                         next.set);
  TD_CUDA(cudaGetLastError());
  return TD_OK;
}

// One instantiation of the attention kernels per (layout, P precision).
template <bool kPaged, bool kSplit>
cudaError_t launch_attn_kernel(const AttnPlan& a, int D, const CUtensorMap& mq,
                               const CUtensorMap& mkc, const CUtensorMap& mvc,
                               const CUtensorMap& mkb, const CUtensorMap& mvb,
                               const AttnParams& p, cudaStream_t st) {
  if (a.pair) {
    auto k = attn_pair_kernel<kPaged, kSplit>;
    cudaError_t e = set_smem(k, PairSmem::kBytes);
    if (e != cudaSuccess) return e;
    k<<<a.ncta, kAttnThreads, PairSmem::kBytes, st>>>(mq, mkc, mvc, mkb, mvb, p);
  } else if (D == 128) {
    auto k = attn_fused_kernel<128, kPaged, kSplit>;
    cudaError_t e = set_smem(k, AttnSmem<128>::kBytes);
    if (e != cudaSuccess) return e;
    k<<<a.ncta, kAttnThreads, AttnSmem<128>::kBytes, st>>>(mq, mkc, mvc, mkb, mvb, p);
  } else {
    auto k = attn_fused_kernel<64, kPaged, kSplit>;
    cudaError_t e = set_smem(k, AttnSmem<64>::kBytes);
    if (e != cudaSuccess) return e;
    k<<<a.ncta, kAttnThreads, AttnSmem<64>::kBytes, st>>>(mq, mkc, mvc, mkb, mvb, p);
  }
  return cudaGetLastError();
}

td_status run_attention(const td_dims* dm, const void* q, const void* k_blk, const void* v_blk,
                        const void* k_ctx, const void* v_ctx, const int* ctx_len,
                        const td_paging* pg, int precision, void* o, float* lse, void* ws,
                        cudaStream_t st, int nsm, const int* skip = nullptr) {
  const bool paged = pg != nullptr && pg->page_table != nullptr;
  const AttnPlan a = plan_attention(dm, nsm);
  const int D = dm->D;
  CUtensorMap mq, mkc, mvc, mkb, mvb;
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)dm->Hq, (uint64_t)dm->S, (uint64_t)dm->B};
    const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)dm->Hq * D * 2,
                             (uint64_t)dm->S * dm->Hq * D * 2};
    const uint32_t box[4] = {64, (uint32_t)a.Gc, (uint32_t)dm->S, 1};
    if (!make_map(&mq, q, 4, dims, str, box)) return TD_ERR_CUDA;
  }
  // K/V boxes: the single-SM kernel loads whole 128-key tiles (block keys: S rows); the pair
  // kernel loads its half: 64 keys of K, 64 head dims of V (block keys: 64 / 128 rows, the
  // rows beyond S lie outside the tensor and arrive as zeros)
  const uint32_t kb_rows = a.pair ? 64 : kKeyTile, vb_rows = kKeyTile;
  const uint32_t blk_k = a.pair ? 64 : (uint32_t)dm->S, blk_v = a.pair ? 128 : (uint32_t)dm->S;
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)dm->Hkv, (uint64_t)dm->S, (uint64_t)dm->B};
    const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)dm->Hkv * D * 2,
                             (uint64_t)dm->S * dm->Hkv * D * 2};
    const uint32_t boxk[4] = {64, 1, blk_k, 1};
    const uint32_t boxv[4] = {64, 1, blk_v, 1};
    if (!make_map(&mkb, k_blk, 4, dims, str, boxk) || !make_map(&mvb, v_blk, 4, dims, str, boxv))
      return TD_ERR_CUDA;
  }
  {
    // an empty cache still needs a well-formed (never used) descriptor; a paged cache is one
    // [128][D] slab per (page, KV head)
    const bool empty = dm->Lmax == 0;
    const uint64_t rows = empty ? 1 : (paged ? (uint64_t)kKeyTile : (uint64_t)dm->Lmax);
    const uint64_t slabs =
        empty ? 1 : (paged ? (uint64_t)pg->n_pages * dm->Hkv : (uint64_t)dm->B * dm->Hkv);
    const uint64_t dims[3] = {(uint64_t)D, rows, slabs};
    const uint64_t str[2] = {(uint64_t)D * 2, rows * D * 2};
    const uint32_t boxk[3] = {64, kb_rows, 1};
    const uint32_t boxv[3] = {64, vb_rows, 1};
    const void* kb = empty ? k_blk : k_ctx;
    const void* vb = empty ? v_blk : v_ctx;
    if (!make_map(&mkc, kb, 3, dims, str, boxk) || !make_map(&mvc, vb, 3, dims, str, boxv))
      return TD_ERR_CUDA;
  }
  AttnParams p{};
  p.B = dm->B; p.S = dm->S; p.Hq = dm->Hq; p.Hkv = dm->Hkv; p.D = D; p.Lmax = dm->Lmax;
  p.G = a.G; p.Gc = a.Gc; p.NC = a.NC; p.NCT = a.NCT; p.R = a.R;
  p.n_ctx_tiles = a.n_ctx_tiles; p.T = a.T; p.n_units = a.n_units; p.n_teams = a.n_teams;
  p.total = a.total;
  p.max_seg = a.max_seg;
  p.ctx_len = ctx_len;
  p.q = static_cast<const uint16_t*>(q);
  p.skip = skip;
  p.page_table = paged ? pg->page_table : nullptr;
  p.max_pages = paged ? pg->max_pages : 0;
  p.n_pages = paged ? pg->n_pages : 0;
  p.part_o = static_cast<float*>(ws);
  p.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + a.part_o_bytes);
  p.out = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  const bool split = precision == TD_ATTN_P_SPLIT;
  cudaError_t ke;
  if (paged)
    ke = split ? launch_attn_kernel<true, true>(a, D, mq, mkc, mvc, mkb, mvb, p, st)
               : launch_attn_kernel<true, false>(a, D, mq, mkc, mvc, mkb, mvb, p, st);
  else
    ke = split ? launch_attn_kernel<false, true>(a, D, mq, mkc, mvc, mkb, mvb, p, st)
               : launch_attn_kernel<false, false>(a, D, mq, mkc, mvc, mkb, mvb, p, st);
  TD_CUDA(ke);
  if (a.split) {
    const dim3 grid(a.n_units * a.NC, (a.R + kMergeRows - 1) / kMergeRows);
    attn_merge_kernel<<<grid, kMergeRows * (D / 4), 0, st>>>(p);
    TD_CUDA(cudaGetLastError());
  }
  return TD_OK;
}

// ------------------------------------------------------------------------------------------
// Denoise-step workspace
// ------------------------------------------------------------------------------------------
struct StepWs {
  uint16_t *h, *xmod, *q, *k, *v, *o;
  float2* rope;     // [B*S][D/2] (cos, sin) of the rotary variant
  uint16_t* h_lm;   // last layer's output, rows masked at the step start only (compacted)
  int* row_pos;     // [B*S] compact index of each row, -1 if committed
  int* m_count;     // number of rows in h_lm
  float* gate;
  void* attn;
  void* lm;
  int* loop;      // decode-loop step counter
  size_t total;
};

StepWs carve_step(const td_dims* dm, void* base, int nsm) {
  StepWs w{};
  const size_t M = (size_t)dm->B * dm->S;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  const size_t o_h = take(M * dm->d * 2), o_x = take(M * dm->d * 2);
  const size_t o_q = take(M * dm->Hq * dm->D * 2), o_k = take(M * dm->Hkv * dm->D * 2),
               o_v = take(M * dm->Hkv * dm->D * 2), o_o = take(M * dm->Hq * dm->D * 2);
  const size_t o_hl = take(M * dm->d * 2), o_rp = take(M * 4), o_mc = take(16);
  const size_t o_ro = take(M * (size_t)(dm->D / 2) * sizeof(float2));
  const size_t o_g = take((size_t)dm->d * 4);
  const size_t o_a = take(attn_ws_bytes(dm, nsm));
  const size_t o_l = take(lm_ws_bytes((int)M, dm->V));
  const size_t o_c = take(64);
  w.total = off;
  if (base) {
    uint8_t* b = static_cast<uint8_t*>(base);
    w.h = reinterpret_cast<uint16_t*>(b + o_h);
    w.xmod = reinterpret_cast<uint16_t*>(b + o_x);
    w.q = reinterpret_cast<uint16_t*>(b + o_q);
    w.k = reinterpret_cast<uint16_t*>(b + o_k);
    w.v = reinterpret_cast<uint16_t*>(b + o_v);
    w.o = reinterpret_cast<uint16_t*>(b + o_o);
    w.h_lm = reinterpret_cast<uint16_t*>(b + o_hl);
    w.rope = reinterpret_cast<float2*>(b + o_ro);
    w.row_pos = reinterpret_cast<int*>(b + o_rp);
    w.m_count = reinterpret_cast<int*>(b + o_mc);
    w.gate = reinterpret_cast<float*>(b + o_g);
    w.attn = b + o_a;
    w.lm = b + o_l;
    w.loop = reinterpret_cast<int*>(b + o_c);
  }
  return w;
}

td_status run_step(const td_dims* dm, const td_layer* layers, const int* ctx_len, const void* h,
                   const void* emb, const void* pos, const void* w_lm, const float* phi_t,
                   int t, int T, float gamma, int rule, float rope_theta,
                   const td_paging* paging, int precision, int* tokens, unsigned char* masked,
                   float* conf, int* pred, int* n_committed, int* all_done, void* ws,
                   cudaStream_t st, int nsm, const int* skip = nullptr, int* steps = nullptr,
                   void* h_out = nullptr, const NextStep& next = NextStep{}) {
  const StepWs w = carve_step(dm, ws, nsm);
  const int M = dm->B * dm->S;
  const int d = dm->d;
  if (h == nullptr) {
    embed_kernel<<<M, 256, 0, st>>>(tokens, static_cast<const uint16_t*>(emb),
                                    static_cast<const uint16_t*>(pos), w.h, dm->S, d, dm->V,
                                    skip);
  } else {
    TD_CUDA(cudaMemcpyAsync(w.h, h, (size_t)M * d * 2, cudaMemcpyDeviceToDevice, st));
  }
  TD_CUDA(cudaGetLastError());
  // the LM head evaluates only the rows still masked now: the last layer writes them,
  // compacted, into h_lm
  const int first_only = (rule == kRuleLeftToRight && t != T) ? 1 : 0;
  lm_rows_kernel<<<1, kRowsThreads, 0, st>>>(masked, M, dm->S, first_only, w.row_pos,
                                             w.m_count, skip);
  TD_CUDA(cudaGetLastError());
  const int nq = dm->Hq * dm->D, nk = dm->Hkv * dm->D;
  const int bn = M >= 512 ? 256 : 128;
  if (rope_theta > 0.f) {
    const int total = M * (dm->D / 2);
    rope_table_kernel<<<(total + 255) / 256, 256, 0, st>>>(ctx_len, dm->B, dm->S, dm->Lmax, dm->D,
                                                          (double)rope_theta, w.rope, skip);
    TD_CUDA(cudaGetLastError());
  }
  for (int l = 0; l < dm->n_layers; ++l) {
    const td_layer& L = layers[l];
    td_status sa = launch_adaln(w.h, L.ada_E, phi_t, M, d, kLnEps, w.xmod, w.gate, st, skip);
    if (sa != TD_OK) return sa;
    GemmParams g1{};
    g1.q = w.q; g1.k = w.k; g1.v = w.v; g1.nq = nq; g1.nk = nk; g1.skip = skip;
    g1.rope_cs = w.rope;
    g1.head_dim = dm->D;
    td_status s =
        rope_theta > 0.f
            ? gemm_dispatch<EPI_QKV_ROPE>(w.xmod, L.wqkv, M, nq + 2 * nk, d, g1, st, nsm, bn)
            : gemm_dispatch<EPI_QKV>(w.xmod, L.wqkv, M, nq + 2 * nk, d, g1, st, nsm, bn);
    if (s != TD_OK) return s;
    s = run_attention(dm, w.q, w.k, w.v, L.k_ctx, L.v_ctx, ctx_len, paging, precision, w.o,
                      nullptr, w.attn, st, nsm, skip);
    if (s != TD_OK) return s;
    GemmParams g2{};
    g2.h = w.h; g2.gate = w.gate; g2.skip = skip;
    if (l == dm->n_layers - 1 && h_out == nullptr) {
      // the last layer writes only the rows the LM head evaluates, compacted
      g2.row_pos = w.row_pos;
      g2.h_out = w.h_lm;
    }
    s = gemm_dispatch<EPI_RESID>(w.o, L.wo, M, d, nq, g2, st, nsm, bn);
    if (s != TD_OK) return s;
  }
  if (dm->n_layers == 0 || h_out != nullptr) {
    // every row of the final hidden state is in w.h: report it if asked, then gather the
    // rows the LM head evaluates (the same values the compacted epilogue writes)
    if (h_out != nullptr)
      TD_CUDA(cudaMemcpyAsync(h_out, w.h, (size_t)M * d * 2, cudaMemcpyDeviceToDevice, st));
    gather_rows_kernel<<<M, 256, 0, st>>>(w.h, w.row_pos, w.h_lm, d, skip);
    TD_CUDA(cudaGetLastError());
  }
  return run_lmhead_commit(dm, w.h_lm, w_lm, gamma, rule, t == T ? 1 : 0, tokens, masked, conf,
                           pred,
                           n_committed, all_done, w.lm, st, nsm, skip, steps, w.row_pos,
                           w.m_count, next);
}

td_status check_layers(const td_dims* dm, const td_layer* layers) {
  if (dm->n_layers > 0 && !layers) return TD_ERR_INVALID_ARG;
  for (int l = 0; l < dm->n_layers; ++l) {
    const td_layer& L = layers[l];
    if (!L.wqkv || !L.wo || !L.ada_E) return TD_ERR_INVALID_ARG;
    if (dm->Lmax > 0 && (!L.k_ctx || !L.v_ctx)) return TD_ERR_INVALID_ARG;
    if (!aligned16(L.wqkv) || !aligned16(L.wo) || !aligned16(L.ada_E) ||
        (dm->Lmax > 0 && (!aligned16(L.k_ctx) || !aligned16(L.v_ctx))))
      return TD_ERR_INVALID_ARG;
  }
  return TD_OK;
}

// ------------------------------------------------------------------------------------------
// Decode loop as one CUDA graph: the T steps are captured once per distinct argument set (on
// a private stream, since the legacy default stream cannot be captured) and replayed on the
// caller's stream. Each step sits in a conditional node that runs only while positions are
// left (see build_loop_conditional); every kernel also reads the all-done word that the
// previous step's commit wrote and returns at once when it is set, which is what ends the
// loop in the flat graph used where conditional nodes are unavailable. merge_commit counts
// the steps that ran.
// ------------------------------------------------------------------------------------------
void set_all_smem() {
  set_smem(gemm_tn_kernel<128, 6, EPI_QKV>, GemmSmem<128, 6>::kBytes);
  set_smem(gemm_tn_kernel<128, 6, EPI_RESID>, GemmSmem<128, 6>::kBytes);
  set_smem(gemm_tn_kernel<128, 6, EPI_LMHEAD>, GemmSmem<128, 6>::kBytes);
  set_smem(gemm_tn_kernel<128, 6, EPI_QKV_ROPE>, GemmSmem<128, 6>::kBytes);
  constexpr int sq = pair_gemm_stages(EPI_QKV), sr = pair_gemm_stages(EPI_RESID);
  constexpr int sl = pair_gemm_stages(EPI_LMHEAD), sp = pair_gemm_stages(EPI_QKV_ROPE);
  set_smem(gemm_pair_kernel<sq, EPI_QKV>, GemmPairSmem<sq, EPI_QKV>::kBytes);
  set_smem(gemm_pair_kernel<sr, EPI_RESID>, GemmPairSmem<sr, EPI_RESID>::kBytes);
  set_smem(gemm_pair_kernel<sl, EPI_LMHEAD>, GemmPairSmem<sl, EPI_LMHEAD>::kBytes);
  set_smem(gemm_pair_kernel<sp, EPI_QKV_ROPE>, GemmPairSmem<sp, EPI_QKV_ROPE>::kBytes);
  set_smem(attn_fused_kernel<128, false, false>, AttnSmem<128>::kBytes);
  set_smem(attn_fused_kernel<64, false, false>, AttnSmem<64>::kBytes);
  set_smem(attn_pair_kernel<false, false>, PairSmem::kBytes);
  set_smem(attn_fused_kernel<128, true, false>, AttnSmem<128>::kBytes);
  set_smem(attn_fused_kernel<64, true, false>, AttnSmem<64>::kBytes);
  set_smem(attn_pair_kernel<true, false>, PairSmem::kBytes);
  set_smem(attn_fused_kernel<128, false, true>, AttnSmem<128>::kBytes);
  set_smem(attn_fused_kernel<64, false, true>, AttnSmem<64>::kBytes);
  set_smem(attn_pair_kernel<false, true>, PairSmem::kBytes);
  set_smem(attn_fused_kernel<128, true, true>, AttnSmem<128>::kBytes);
  set_smem(attn_fused_kernel<64, true, true>, AttnSmem<64>::kBytes);
  set_smem(attn_pair_kernel<true, true>, PairSmem::kBytes);
}

struct LoopKey {
  std::vector<uint64_t> v;
  bool operator<(const LoopKey& o) const { return v < o.v; }
};

std::mutex g_loop_mu;
std::atomic<int> g_loop_form_wanted{1};   // 1 conditional nodes, 2 flat
std::atomic<int> g_loop_form_built{0};
std::map<LoopKey, cudaGraphExec_t> g_loop_graphs;
std::vector<LoopKey> g_loop_order;
constexpr size_t kMaxLoopGraphs = 16;

cudaStream_t capture_stream() {
  static std::mutex mu;
  static std::map<int, cudaStream_t> streams;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  auto it = streams.find(dev);
  if (it != streams.end()) return it->second;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
  streams[dev] = s;
  return s;
}

// The loop as a chain of conditional (if) nodes, one per step: the first step's condition
// defaults to 1 at every launch, the others to 0, and the commit kernel of step t sets the
// condition of step t+1 to "positions left", so the steps after the one that committed the
// block's last position launch nothing. Each step's kernels are captured into its node's body.
// TD_ERR_UNSUPPORTED: conditional nodes are not available (the caller builds the flat graph).
td_status build_loop_conditional(const td_dims* dm, const td_layer* layers, const int* ctx_len,
                                 const void* emb, const void* pos, const void* w_lm,
                                 const float* phi_table, int t_start, int T, float gamma,
                                 int rule, float rope_theta, const td_paging* paging,
                                 int precision, int* tokens, unsigned char* masked, float* conf,
                                 int* pred, int* n_committed, int* all_done, void* ws,
                                 const StepWs& w, cudaStream_t cs, int nsm, cudaGraph_t* out) {
  cudaGraph_t g = nullptr;
  if (cudaGraphCreate(&g, 0) != cudaSuccess) {
    cudaGetLastError();
    return TD_ERR_UNSUPPORTED;
  }
  std::vector<cudaGraphConditionalHandle> cond(T - t_start + 1);
  for (int t = t_start; t <= T; ++t) {
    if (cudaGraphConditionalHandleCreate(&cond[t - t_start], g, t == t_start ? 1u : 0u,
                                         cudaGraphCondAssignDefault) != cudaSuccess) {
      cudaGraphDestroy(g);
      cudaGetLastError();
      return TD_ERR_UNSUPPORTED;
    }
  }
  cudaGraphNode_t prev = nullptr;
  for (int t = t_start; t <= T; ++t) {
    cudaGraphNodeParams np{};
    np.type = cudaGraphNodeTypeConditional;
    np.conditional.handle = cond[t - t_start];
    np.conditional.type = cudaGraphCondTypeIf;
    np.conditional.size = 1;
    cudaGraphNode_t node = nullptr;
    if (cudaGraphAddNode(&node, g, prev ? &prev : nullptr, nullptr, prev ? 1 : 0, &np) !=
        cudaSuccess) {
      cudaGraphDestroy(g);
      cudaGetLastError();
      return TD_ERR_UNSUPPORTED;
    }
    prev = node;
    cudaGraph_t body = np.conditional.phGraph_out[0];
    if (cudaStreamBeginCaptureToGraph(cs, body, nullptr, nullptr, 0,
                                      cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      cudaGraphDestroy(g);
      cudaGetLastError();
      return TD_ERR_UNSUPPORTED;
    }
    td_status s = TD_OK;
    if (t == t_start && (cudaMemsetAsync(all_done, 0, sizeof(int), cs) != cudaSuccess ||
                         cudaMemsetAsync(w.loop, 0, sizeof(int), cs) != cudaSuccess))
      s = TD_ERR_CUDA;
    NextStep next;
    if (t < T) {
      next.handle = cond[t + 1 - t_start];
      next.set = 1;
    }
    if (s == TD_OK)
      s = run_step(dm, layers, ctx_len, nullptr, emb, pos, w_lm,
                   phi_table + (size_t)(t - 1) * 6 * dm->d, t, T, gamma, rule, rope_theta,
                   paging, precision, tokens, masked, conf, pred, n_committed, all_done, ws, cs,
                   nsm, all_done, w.loop, nullptr, next);
    cudaGraph_t captured = nullptr;
    const cudaError_t ee = cudaStreamEndCapture(cs, &captured);
    if (s != TD_OK || ee != cudaSuccess) {
      cudaGraphDestroy(g);
      cudaGetLastError();
      return s != TD_OK ? s : TD_ERR_UNSUPPORTED;
    }
  }
  *out = g;
  return TD_OK;
}

// The loop as one flat capture of all T steps; every kernel of step t+1 reads the all-done
// word that step t's commit wrote and returns at once when it is set.
td_status build_loop_flat(const td_dims* dm, const td_layer* layers, const int* ctx_len,
                          const void* emb, const void* pos, const void* w_lm,
                          const float* phi_table, int t_start, int T, float gamma, int rule,
                          float rope_theta, const td_paging* paging, int precision, int* tokens,
                          unsigned char* masked, float* conf, int* pred, int* n_committed,
                          int* all_done, void* ws, const StepWs& w, cudaStream_t cs, int nsm,
                          cudaGraph_t* out) {
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return TD_ERR_UNSUPPORTED;
  }
  td_status s = TD_OK;
  if (cudaMemsetAsync(all_done, 0, sizeof(int), cs) != cudaSuccess ||
      cudaMemsetAsync(w.loop, 0, sizeof(int), cs) != cudaSuccess)
    s = TD_ERR_CUDA;
  for (int t = t_start; t <= T && s == TD_OK; ++t)
    s = run_step(dm, layers, ctx_len, nullptr, emb, pos, w_lm,
                 phi_table + (size_t)(t - 1) * 6 * dm->d, t, T, gamma, rule, rope_theta, paging,
                 precision, tokens, masked, conf, pred, n_committed, all_done, ws, cs, nsm,
                 all_done, w.loop);
  cudaGraph_t g = nullptr;
  const cudaError_t ee = cudaStreamEndCapture(cs, &g);
  if (s != TD_OK || ee != cudaSuccess || g == nullptr) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return s != TD_OK ? s : TD_ERR_UNSUPPORTED;
  }
  *out = g;
  return TD_OK;
}

// Runs the loop through a cached graph. TD_ERR_UNSUPPORTED means "capture not possible here":
// the caller then runs the host loop.
td_status decode_graph(const td_dims* dm, const td_layer* layers, const int* ctx_len,
                       const void* emb, const void* pos, const void* w_lm,
                       const float* phi_table, int t_start, int T, float gamma, int rule,
                       float rope_theta, const td_paging* paging, int precision, int* tokens,
                       unsigned char* masked, float* conf, int* pred,
                       int* n_committed, int* all_done, void* ws, size_t ws_bytes,
                       cudaStream_t st, int nsm, int* steps_taken, int* done) {
  const StepWs w = carve_step(dm, ws, nsm);
  LoopKey key;
  int dev = 0;
  TD_CUDA(cudaGetDevice(&dev));
  auto u = [&](const void* p) { key.v.push_back(reinterpret_cast<uintptr_t>(p)); };
  key.v = {(uint64_t)dev, (uint64_t)dm->B, (uint64_t)dm->S, (uint64_t)dm->d, (uint64_t)dm->Hq,
           (uint64_t)dm->Hkv, (uint64_t)dm->D, (uint64_t)dm->V, (uint64_t)dm->Lmax,
           (uint64_t)dm->n_layers, (uint64_t)t_start, (uint64_t)T, (uint64_t)ws_bytes};
  uint32_t gbits;
  std::memcpy(&gbits, &gamma, 4);
  key.v.push_back(gbits);
  key.v.push_back((uint64_t)rule);
  uint32_t rbits;
  std::memcpy(&rbits, &rope_theta, 4);
  key.v.push_back(rbits);
  u(paging ? paging->page_table : nullptr);
  key.v.push_back((uint64_t)precision);
  key.v.push_back(paging ? (uint64_t)paging->max_pages : 0);
  key.v.push_back(paging ? (uint64_t)paging->n_pages : 0);
  for (int l = 0; l < dm->n_layers; ++l) {
    u(layers[l].wqkv); u(layers[l].wo); u(layers[l].ada_E); u(layers[l].k_ctx); u(layers[l].v_ctx);
  }
  u(ctx_len); u(emb); u(pos); u(w_lm); u(phi_table); u(tokens); u(masked); u(conf); u(pred);
  u(n_committed); u(all_done); u(ws);
  const int form_wanted = g_loop_form_wanted.load();
  key.v.push_back((uint64_t)form_wanted);
  {
    // One lock over lookup, capture, insertion and launch: no two threads capture on the
    // shared capture stream at once, a key is captured once, and no graph is destroyed
    // between its lookup and its launch (eviction synchronizes the device first, so launches
    // already queued finish before their graph goes).
    std::lock_guard<std::mutex> lk(g_loop_mu);
    cudaGraphExec_t exec = nullptr;
    auto it = g_loop_graphs.find(key);
    if (it != g_loop_graphs.end()) exec = it->second;
    if (exec == nullptr) {
      set_all_smem();
      cudaStream_t cs = capture_stream();
      if (cs == nullptr) return TD_ERR_UNSUPPORTED;
      // the chain of conditional nodes first; the flat capture where that cannot be built
      // or instantiated
      for (int flat = form_wanted == 2 ? 1 : 0; flat < 2 && exec == nullptr; ++flat) {
        cudaGraph_t g = nullptr;
        const td_status s =
            flat == 0
                ? build_loop_conditional(dm, layers, ctx_len, emb, pos, w_lm, phi_table,
                                         t_start, T, gamma, rule, rope_theta, paging, precision,
                                         tokens, masked, conf, pred, n_committed, all_done, ws,
                                         w, cs, nsm, &g)
                : build_loop_flat(dm, layers, ctx_len, emb, pos, w_lm, phi_table, t_start, T,
                                  gamma, rule, rope_theta, paging, precision, tokens, masked,
                                  conf, pred, n_committed, all_done, ws, w, cs, nsm, &g);
        if (s == TD_ERR_UNSUPPORTED) continue;
        if (s != TD_OK) return s;
        if (cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) {
          exec = nullptr;
          cudaGetLastError();
        } else {
          g_loop_form_built.store(flat ? 2 : 1);
        }
        cudaGraphDestroy(g);
      }
      if (exec == nullptr) return TD_ERR_UNSUPPORTED;
      g_loop_graphs[key] = exec;
      g_loop_order.push_back(key);
      if (g_loop_order.size() > kMaxLoopGraphs) {
        auto old = g_loop_graphs.find(g_loop_order.front());
        if (old != g_loop_graphs.end()) {
          cudaDeviceSynchronize();
          cudaGraphExecDestroy(old->second);
          g_loop_graphs.erase(old);
        }
        g_loop_order.erase(g_loop_order.begin());
      }
    }
    TD_CUDA(cudaGraphLaunch(exec, st));
  }
  int host[2] = {0, 0};
  TD_CUDA(cudaMemcpyAsync(&host[0], w.loop, sizeof(int), cudaMemcpyDeviceToHost, st));
  TD_CUDA(cudaMemcpyAsync(&host[1], all_done, sizeof(int), cudaMemcpyDeviceToHost, st));
  TD_CUDA(cudaStreamSynchronize(st));
  *steps_taken = host[0];
  *done = host[1];
  return TD_OK;
}

bool rule_ok(int rule) {
  return rule == TD_COMMIT_CONFIDENCE || rule == TD_COMMIT_LEFT_TO_RIGHT;
}

// A paged layout must cover every sequence's Lmax and name a non-empty pool.
bool paging_ok(const td_dims* dm, const td_paging* pg) {
  if (pg == nullptr || pg->page_table == nullptr) return true;
  const long long tiles = ((long long)dm->Lmax + kKeyTile - 1) / kKeyTile;
  return pg->n_pages >= 1 && pg->max_pages >= tiles && pg->max_pages >= 1 &&
         (long long)pg->n_pages * dm->Hkv < (1ll << 31);
}

// Options of a step (NULL: confidence masking, no rotation, contiguous caches); false if
// they are invalid.
bool precision_ok(int precision) {
  return precision == TD_ATTN_P_BF16 || precision == TD_ATTN_P_SPLIT;
}

bool read_opts(const td_dims* dm, const td_step_opts* opts, int* rule, float* rope_theta,
               const td_paging** paging, void** h_out, int* precision) {
  *rule = opts ? opts->rule : TD_COMMIT_CONFIDENCE;
  *rope_theta = opts ? opts->rope_theta : 0.f;
  *paging = (opts && opts->paging.page_table) ? &opts->paging : nullptr;
  *h_out = opts ? opts->h_out : nullptr;
  *precision = opts ? opts->attn_precision : TD_ATTN_P_BF16;
  return rule_ok(*rule) && std::isfinite(*rope_theta) && *rope_theta >= 0.f &&
         paging_ok(dm, *paging) && (*h_out == nullptr || aligned16(*h_out)) &&
         precision_ok(*precision);
}

bool ws_ok(const void* ws, size_t have, size_t need) {
  if (need == 0) return true;
  return ws != nullptr && have >= need && (reinterpret_cast<uintptr_t>(ws) % kAlign) == 0;
}

}  // namespace

// ==========================================================================================
// C ABI
// ==========================================================================================
extern "C" {

const char* td_status_string(td_status s) {
  switch (s) {
    case TD_OK: return "TD_OK";
    case TD_ERR_INVALID_ARG: return "TD_ERR_INVALID_ARG";
    case TD_ERR_WORKSPACE: return "TD_ERR_WORKSPACE";
    case TD_ERR_UNSUPPORTED: return "TD_ERR_UNSUPPORTED";
    case TD_ERR_CUDA: return "TD_ERR_CUDA";
    case TD_ERR_NOT_CONVERGED: return "TD_ERR_NOT_CONVERGED";
    case TD_ERR_DEVICE_TIMEOUT: return "TD_ERR_DEVICE_TIMEOUT";
  }
  return "TD_STATUS_UNKNOWN";
}

size_t td_workspace_size(const td_dims* dm, int fn) {
  const int nsm = sm_count();
  switch (fn) {
    case TD_FN_ADALN_MODULATE:
      return 0;
    case TD_FN_BLOCK_ATTENTION:
      if (check_dims(dm, false) != TD_OK) return (size_t)-1;
      return attn_ws_bytes(dm, nsm);
    case TD_FN_LMHEAD_COMMIT:
      if (check_lm_dims(dm) != TD_OK) return (size_t)-1;
      return lm_ws_bytes(dm->B * dm->S, dm->V);
    case TD_FN_DENOISE_STEP:
    case TD_FN_DECODE_BLOCK:
      if (check_dims(dm, true) != TD_OK) return (size_t)-1;
      return carve_step(dm, nullptr, nsm).total;
  }
  return (size_t)-1;
}

td_status td_adaln_modulate(const void* h, const float* E, const float* phi, int rows, int d,
                            float eps, void* x_mod, void* stream) {
  if (!h || !E || !phi || !x_mod || rows <= 0 || d <= 0 || !(eps >= 0.f))
    return TD_ERR_INVALID_ARG;
  if (d % 8 != 0 || d > kAdaMaxD) return TD_ERR_UNSUPPORTED;
  if (!aligned16(h) || !aligned16(x_mod)) return TD_ERR_INVALID_ARG;
  return launch_adaln(h, E, phi, rows, d, eps, x_mod, nullptr, (cudaStream_t)stream);
}

td_status td_block_attention(const td_dims* dims, const void* q, const void* k_blk,
                             const void* v_blk, const void* k_ctx, const void* v_ctx,
                             const int* ctx_len, const td_paging* paging, int precision,
                             void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
  td_status s = check_dims(dims, false);
  if (s != TD_OK) return s;
  if (!paging_ok(dims, paging) || !precision_ok(precision)) return TD_ERR_INVALID_ARG;
  if (!q || !k_blk || !v_blk || !o) return TD_ERR_INVALID_ARG;
  if (dims->Lmax > 0 && (!k_ctx || !v_ctx)) return TD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_blk) || !aligned16(v_blk) || !aligned16(o) ||
      (dims->Lmax > 0 && (!aligned16(k_ctx) || !aligned16(v_ctx))))
    return TD_ERR_INVALID_ARG;
  const int nsm = sm_count();
  if (!ws_ok(ws, ws_bytes, attn_ws_bytes(dims, nsm))) return TD_ERR_WORKSPACE;
  return run_attention(dims, q, k_blk, v_blk, k_ctx, v_ctx, ctx_len, paging, precision, o, lse,
                       ws, (cudaStream_t)stream, nsm);
}

td_status td_lmhead_commit(const td_dims* dims, const void* h, const void* w_lm, float gamma,
                           int rule, int force_all, int* tokens, unsigned char* masked,
                           float* conf, int* pred, int* n_committed, int* all_done, void* ws,
                           size_t ws_bytes, void* stream) {
  td_status s = check_lm_dims(dims);
  if (s != TD_OK) return s;
  if (!rule_ok(rule)) return TD_ERR_INVALID_ARG;
  if (!h || !w_lm || !tokens || !masked || !conf || !pred || !n_committed || !all_done)
    return TD_ERR_INVALID_ARG;
  if (std::isnan(gamma)) return TD_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w_lm)) return TD_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, lm_ws_bytes(dims->B * dims->S, dims->V))) return TD_ERR_WORKSPACE;
  return run_lmhead_commit(dims, h, w_lm, gamma, rule, force_all, tokens, masked, conf, pred,
                           n_committed, all_done, ws, (cudaStream_t)stream, sm_count());
}

td_status td_denoise_step(const td_dims* dims, const td_layer* layers, const int* ctx_len,
                          const void* h, const void* emb, const void* pos, const void* w_lm,
                          const float* phi_t, int t, int T, float gamma,
                          const td_step_opts* opts, int* tokens, unsigned char* masked,
                          float* conf, int* pred, int* n_committed, int* all_done, void* ws,
                          size_t ws_bytes, void* stream) {
  td_status s = check_dims(dims, true);
  if (s != TD_OK) return s;
  int rule = 0;
  float rope_theta = 0.f;
  const td_paging* paging = nullptr;
  void* h_out = nullptr;
  int precision = 0;
  if (!read_opts(dims, opts, &rule, &rope_theta, &paging, &h_out, &precision))
    return TD_ERR_INVALID_ARG;
  if ((s = check_layers(dims, layers)) != TD_OK) return s;
  if (!w_lm || !phi_t || !tokens || !masked || !conf || !pred || !n_committed || !all_done)
    return TD_ERR_INVALID_ARG;
  if (!h && (!emb || !pos)) return TD_ERR_INVALID_ARG;
  // emb / pos are read in 16-byte vectors, w_lm through a tensor map
  if (!aligned16(w_lm) || (!h && (!aligned16(emb) || !aligned16(pos))))
    return TD_ERR_INVALID_ARG;
  if (t < 1 || T < 1 || t > T || std::isnan(gamma)) return TD_ERR_INVALID_ARG;
  const int nsm = sm_count();
  if (!ws_ok(ws, ws_bytes, carve_step(dims, nullptr, nsm).total)) return TD_ERR_WORKSPACE;
  return run_step(dims, layers, ctx_len, h, emb, pos, w_lm, phi_t, t, T, gamma, rule,
                  rope_theta, paging, precision, tokens, masked,
                  conf, pred, n_committed, all_done, ws, (cudaStream_t)stream, nsm, nullptr,
                  nullptr, h_out);
}

td_status td_decode_block(const td_dims* dims, const td_layer* layers, const int* ctx_len,
                          const void* emb, const void* pos, const void* w_lm,
                          const float* phi_table, int t_start, int T, float gamma,
                          const td_step_opts* opts, int* tokens, unsigned char* masked,
                          float* conf, int* pred, int* n_committed, int* all_done,
                          int* steps_taken, void* ws, size_t ws_bytes, void* stream) {
  td_status s = check_dims(dims, true);
  if (s != TD_OK) return s;
  int rule = 0;
  float rope_theta = 0.f;
  const td_paging* paging = nullptr;
  void* h_out = nullptr;
  int precision = 0;
  if (!read_opts(dims, opts, &rule, &rope_theta, &paging, &h_out, &precision))
    return TD_ERR_INVALID_ARG;
  if (h_out != nullptr) return TD_ERR_INVALID_ARG;   // a loop has no single final state
  if ((s = check_layers(dims, layers)) != TD_OK) return s;
  if (!emb || !pos || !w_lm || !phi_table || !tokens || !masked || !conf || !pred ||
      !n_committed || !all_done || !steps_taken)
    return TD_ERR_INVALID_ARG;
  if (!aligned16(w_lm) || !aligned16(emb) || !aligned16(pos)) return TD_ERR_INVALID_ARG;
  if (t_start < 1 || T < 1 || std::isnan(gamma)) return TD_ERR_INVALID_ARG;
  const int nsm = sm_count();
  if (!ws_ok(ws, ws_bytes, carve_step(dims, nullptr, nsm).total)) return TD_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  *steps_taken = 0;
  // nothing masked on entry: nothing to do
  {
    std::vector<unsigned char> m((size_t)dims->B * dims->S);
    TD_CUDA(cudaMemcpyAsync(m.data(), masked, m.size(), cudaMemcpyDeviceToHost, st));
    TD_CUDA(cudaStreamSynchronize(st));
    bool any = false;
    for (unsigned char c : m) any |= (c != 0);
    if (!any) return TD_OK;
  }
  int done = 0;
  if (t_start <= T) {
    s = decode_graph(dims, layers, ctx_len, emb, pos, w_lm, phi_table, t_start, T, gamma, rule,
                     rope_theta, paging, precision, tokens, masked, conf, pred, n_committed,
                     all_done, ws, ws_bytes, st, nsm, steps_taken, &done);
    if (s == TD_OK) return done ? TD_OK : TD_ERR_NOT_CONVERGED;
    if (s != TD_ERR_UNSUPPORTED) return s;
  }
  // host loop (when the loop cannot be captured): one all-done read-back per step
  *steps_taken = 0;
  for (int t = t_start; t <= T; ++t) {
    s = run_step(dims, layers, ctx_len, nullptr, emb, pos, w_lm,
                 phi_table + (size_t)(t - 1) * 6 * dims->d, t, T, gamma, rule, rope_theta,
                 paging, precision, tokens, masked, conf, pred, n_committed, all_done, ws, st,
                 nsm);
    if (s != TD_OK) return s;
    TD_CUDA(cudaMemcpyAsync(&done, all_done, sizeof(int), cudaMemcpyDeviceToHost, st));
    TD_CUDA(cudaStreamSynchronize(st));
    ++*steps_taken;
    if (done) break;
  }
  return done ? TD_OK : TD_ERR_NOT_CONVERGED;
}

td_status td_kv_append(const td_dims* dims, const td_layer* layers, const td_kv* block_kv,
                       int* ctx_len, const td_paging* paging, void* stream) {
  td_status s = check_dims(dims, false);
  if (s != TD_OK) return s;
  if (!paging_ok(dims, paging)) return TD_ERR_INVALID_ARG;
  const bool paged = paging != nullptr && paging->page_table != nullptr;
  if (dims->n_layers < 0 || (dims->n_layers > 0 && (!layers || !block_kv)) || !ctx_len)
    return TD_ERR_INVALID_ARG;
  if (dims->Lmax < dims->S) return TD_ERR_INVALID_ARG;   // a block can never fit
  for (int l = 0; l < dims->n_layers; ++l) {
    const td_layer& L = layers[l];
    const td_kv& N = block_kv[l];
    if (!L.k_ctx || !L.v_ctx || !N.k || !N.v) return TD_ERR_INVALID_ARG;
    if (!aligned16(L.k_ctx) || !aligned16(L.v_ctx) || !aligned16(N.k) || !aligned16(N.v))
      return TD_ERR_INVALID_ARG;
  }
  cudaStream_t st = (cudaStream_t)stream;
  const long long chunks = (long long)dims->B * dims->S * dims->Hkv * (dims->D / 8);
  const int threads = 256;
  const int blocks = (int)std::min<long long>((chunks + threads - 1) / threads, 4 * sm_count());
  for (int l = 0; l < dims->n_layers; ++l) {
    // the caches are written here: the const in td_layer is the attention's read-only view
    kv_append_kernel<<<blocks, threads, 0, st>>>(
        static_cast<const uint16_t*>(block_kv[l].k), static_cast<const uint16_t*>(block_kv[l].v),
        static_cast<uint16_t*>(const_cast<void*>(layers[l].k_ctx)),
        static_cast<uint16_t*>(const_cast<void*>(layers[l].v_ctx)), ctx_len, dims->B, dims->S,
        dims->Hkv, dims->D, dims->Lmax, paged ? paging->page_table : nullptr,
        paged ? paging->max_pages : 0, paged ? paging->n_pages : 0);
    TD_CUDA(cudaGetLastError());
  }
  kv_len_update_kernel<<<(dims->B + 255) / 256, 256, 0, st>>>(
      ctx_len, dims->B, dims->S, dims->Lmax, paged ? paging->page_table : nullptr,
      paged ? paging->max_pages : 0, paged ? paging->n_pages : 0);
  TD_CUDA(cudaGetLastError());
  return TD_OK;
}

td_status td_timestep_table(const float* w_t, const float* b_t, int d, int T, float* phi_table,
                            void* stream) {
  if (!w_t || !b_t || !phi_table || d <= 0 || T <= 0 || T > 65536) return TD_ERR_INVALID_ARG;
  if ((long long)6 * d > (1ll << 30)) return TD_ERR_UNSUPPORTED;
  const int rows = 6 * d;
  timestep_table_kernel<<<(rows + kTsWarps - 1) / kTsWarps, 32 * kTsWarps, 0,
                          (cudaStream_t)stream>>>(w_t, b_t, rows, T, phi_table);
  TD_CUDA(cudaGetLastError());
  return TD_OK;
}

int td_decode_graph_form(int form) {
  if (form == 1 || form == 2) g_loop_form_wanted.store(form);
  return g_loop_form_built.load();
}

td_status td_check_bounded_wait(unsigned int limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 2000000u) return TD_ERR_INVALID_ARG;
  wait_check_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(1000ull * limit_us);
  TD_CUDA(cudaGetLastError());
  return TD_OK;
}

td_status td_device_error(int* code) {
  if (!code) return TD_ERR_INVALID_ARG;
  TD_CUDA(cudaDeviceSynchronize());
  unsigned int v = 0, zero = 0;
  TD_CUDA(cudaMemcpyFromSymbol(&v, td::g_error_word, sizeof(v)));
  TD_CUDA(cudaMemcpyToSymbol(td::g_error_word, &zero, sizeof(zero)));
  *code = (int)v;
  // a wait that ran out (TMA, MMA or hand-off) makes the call itself report it
  return (v == td::ERR_WAIT_TMA || v == td::ERR_WAIT_MMA || v == td::ERR_WAIT_EPI)
             ? TD_ERR_DEVICE_TIMEOUT
             : TD_OK;
}

}  // extern "C"

// ==========================================================================================
// td_lmhead_commit_static: the LM head + commit with its scratch in a fixed device array,
// for callers that cannot allocate device memory.
// ==========================================================================================
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr int kMaxDevices = 64;

// The scratch itself. In host code this name is only a stand-in for the device symbol, never
// an address a kernel may use: the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_lm_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device and kept
// for the life of the process (stale after a cudaDeviceReset() of that device).
td_status static_scratch_addr(void** out) {
  int dev = -1;
  TD_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return TD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_addr[dev] == nullptr) {
    void* p = nullptr;
    TD_CUDA(cudaGetSymbolAddress(&p, g_lm_static_scratch));
    if (p == nullptr || (reinterpret_cast<uintptr_t>(p) % kAlign) != 0) return TD_ERR_CUDA;
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return TD_OK;
}

}  // namespace

extern "C" td_status td_lmhead_commit_static(const td_dims* dims, const void* h,
                                             const void* w_lm, float gamma, int force_all,
                                             int* tokens, unsigned char* masked, float* conf,
                                             int* pred, int* n_committed, int* all_done,
                                             void* stream) {
  td_status s = check_lm_dims(dims);
  if (s != TD_OK) return s;
  if (!h || !w_lm || !tokens || !masked || !conf || !pred || !n_committed || !all_done)
    return TD_ERR_INVALID_ARG;
  if (std::isnan(gamma)) return TD_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w_lm)) return TD_ERR_INVALID_ARG;
  if (lm_ws_bytes(dims->B * dims->S, dims->V) > kStaticScratchBytes) return TD_ERR_WORKSPACE;
  void* ws = nullptr;
  if ((s = static_scratch_addr(&ws)) != TD_OK) return s;
  // run_lmhead_commit clears the commit counters in the scratch before the merge kernel.
  return run_lmhead_commit(dims, h, w_lm, gamma, TD_COMMIT_CONFIDENCE, force_all, tokens,
                           masked, conf, pred, n_committed, all_done, ws, (cudaStream_t)stream,
                           sm_count());
}
