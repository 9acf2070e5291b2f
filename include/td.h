/*
 * td.h -- C ABI of the TwoTower block-diffusion denoise step (sm_103a).
 *
 * Sources. The method is described only in prose, on these pages:
 *   [chathome]  "NVIDIA、Nemotron-Labs-TwoTowerを公開：凍結された自己回帰バックボーン上に
 *               構築されたオープンウェイト拡散言語モデル" (news.chathome.org).
 *               Paragraphs used: the inference paragraph ("推論では…": per-layer KV cache,
 *               bidirectional in-block attention, layer-aligned cross-attention, adaLN-single),
 *               the generation paragraph ("生成はブロックごとに…": blocks of S [MASK], T steps,
 *               commit) and the evaluation paragraph ("2×H100 GPUでのBF16評価では…":
 *               confidence masking, threshold gamma = 0.8, block size S = 16).
 *   [aiboss]    "Nemotron-Labs-TwoTower - NVIDIAのオープンソースデュアルタワーアーキテクチャ
 *               普及言語モデル" (aiboss88.com), section "技術原理" (technical principle).
 *   [aikraft]   "Архитектурный прорыв: разделение задач" (aikraft.ru), benchmark paragraph
 *               (gamma = 0.8, S = 16, BF16).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller unless it is documented
 *     as a host pointer. The library never allocates device memory: scratch space is the
 *     caller's `ws` buffer of at least td_workspace_size() bytes, 256-byte aligned.
 *   - bf16 tensors are IEEE bfloat16 stored as uint16; fp32 tensors are IEEE binary32.
 *     All tensors are dense row-major (C order) with the shapes given below; weights are
 *     stored [out_features, in_features] (each output column's weights contiguous).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every call is
 *     asynchronous on it, except td_decode_block, which reads one flag back per step.
 *   - Arguments are validated on the host before anything is launched; a rejected call
 *     launches nothing and returns TD_ERR_INVALID_ARG / TD_ERR_UNSUPPORTED /
 *     TD_ERR_WORKSPACE. No C++ exception crosses this boundary.
 *   - Device-side waits are bounded. A kernel whose wait runs out records a code in a
 *     device error word and returns early; td_device_error() reads (and clears) it.
 *   - Shapes supported by the kernels: D in {64, 128}; Hq % Hkv == 0; 1 <= S <= 64;
 *     d % 64 == 0 (and d <= 8192 for the denoise step); V % 8 == 0; B*S <= 65536;
 *     Lmax >= 0.
 *   - Host threads may call into the library at the same time when their calls use
 *     distinct output and workspace buffers (td_lmhead_commit_static is the exception: all
 *     its calls share one scratch array). The host-side caches (shared-memory opt-ins, the
 *     captured decode graphs) are guarded by locks. The device error word is one per device,
 *     shared by every caller.
 */
#ifndef TD_H_
#define TD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum td_status {
  TD_OK = 0,
  TD_ERR_INVALID_ARG = 1,   /* null pointer, negative/zero size, bad gamma/t/T          */
  TD_ERR_WORKSPACE = 2,     /* ws == NULL or ws_bytes < td_workspace_size(), misaligned */
  TD_ERR_UNSUPPORTED = 3,   /* a shape outside the limits listed above                  */
  TD_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch error, ...)           */
  TD_ERR_NOT_CONVERGED = 5, /* td_decode_block: positions still [MASK] after step T     */
  TD_ERR_DEVICE_TIMEOUT = 6 /* td_device_error: a kernel's bounded wait ran out         */
} td_status;

/* Problem sizes (the pages' notation): B sequences, S block size, d hidden size,
 * Hq query heads, Hkv KV heads (GQA: query head h uses KV head h / (Hq/Hkv)),
 * D head dim, V vocabulary (the [MASK] token id is V, one past the LM-head range),
 * Lmax context KV capacity per sequence, n_layers stacked denoiser attention layers. */
typedef struct td_dims {
  int B, S, d, Hq, Hkv, D, V, Lmax, n_layers;
} td_dims;

/* One denoiser attention layer and the context tower's KV cache of the same layer
 * ([chathome] inference paragraph: each denoiser layer cross-attends to the matching
 * context-tower layer).
 *   wqkv  bf16 [(Hq + 2*Hkv)*D, d]  rows 0..Hq*D-1 = W_q^T, then W_k^T, then W_v^T
 *   wo    bf16 [d, Hq*D]            W_o^T
 *   ada_E fp32 [6, d]               per-layer adaLN-single table E_l (rows: shift, scale,
 *                                   gate, then three rows of the out-of-scope MLP sublayer)
 *   k_ctx bf16 [B, Hkv, Lmax, D]    context keys of this layer (prompt + committed tokens),
 *                                   or a page pool [n_pages, Hkv, 128, D] (td_paging)
 *   v_ctx bf16 [B, Hkv, Lmax, D]    context values of this layer (same layout as k_ctx) */
typedef struct td_layer {
  const void* wqkv;
  const void* wo;
  const float* ada_E;
  const void* k_ctx;
  const void* v_ctx;
} td_layer;

/* Commit rule of a step (the pages name three inference modes of one checkpoint:
 * mask-diffusion, mock-AR and AR-only; [chathome] modes paragraph, [aiboss] overview).
 *   TD_COMMIT_CONFIDENCE    mask-diffusion: confidence masking with threshold gamma
 *                           ([chathome] evaluation paragraph), fallback to the single most
 *                           confident masked position (lowest index on ties).
 *   TD_COMMIT_LEFT_TO_RIGHT mock-AR, a reading (the pages do not define the mode): exactly
 *                           one commit per step, the lowest-index masked position whatever its
 *                           confidence, as AR decoding commits one token per step in order
 *                           ([chathome] generation paragraph). gamma is not used.
 * Both commit every masked position at the last step (force_all / t == T). AR-only mode runs
 * the context tower alone and is outside this library. */
typedef enum td_commit_rule {
  TD_COMMIT_CONFIDENCE = 0,
  TD_COMMIT_LEFT_TO_RIGHT = 1
} td_commit_rule;

/* Paged context cache (optional; NULL or page_table == NULL: contiguous caches).
 * With paging, every layer's k_ctx / v_ctx is a pool of 128-key pages, bf16
 * [n_pages, Hkv, 128, D], and the keys of positions 128 t .. 128 t + 127 of sequence b (its
 * logical context tile t) live in page page_table[b * max_pages + t]. Pages of a sequence need
 * not be contiguous or ordered; sequences may share no page they write. Lmax still bounds every
 * sequence's length (ctx_len[b] <= Lmax), and the entries for its tiles must be in
 * [0, n_pages): an entry outside that range is read as zeros and flags ERR_BAD_PAGE (0x700) in
 * the device error word.
 *   page_table int32 [B, max_pages] device, max_pages >= ceil(Lmax / 128); n_pages >= 1. */
typedef struct td_paging {
  const int* page_table;
  int max_pages;
  int n_pages;
} td_paging;

/* Precision of the softmax probabilities P in the attention's O += P V product (the pages fix
 * no arithmetic beyond BF16; this is a property of this library):
 *   TD_ATTN_P_BF16   P is rounded to bf16 (about 2^-9 relative) for the product: the fast
 *                    default.
 *   TD_ATTN_P_SPLIT  P enters as the sum of two bf16 values, hi = bf16(P) and
 *                    lo = bf16(P - hi) (P carried to about 2^-17 relative), at the cost of a
 *                    second P V product per key tile. Stacked layers then follow an exact
 *                    softmax more closely.
 * Either way the products accumulate in fp32 and the output is rounded to bf16 once. */
typedef enum td_attn_precision {
  TD_ATTN_P_BF16 = 0,
  TD_ATTN_P_SPLIT = 1
} td_attn_precision;

/* Options of a denoise step (td_denoise_step, td_decode_block); NULL means
 * { TD_COMMIT_CONFIDENCE, 0, no paging, NULL, TD_ATTN_P_BF16 }.
 *   rule        a td_commit_rule.
 *   rope_theta  0: no positional rotation (the pages describe none; the embedding path adds
 *               the caller's position table instead). > 0: rotary variant, a reading of a
 *               piece the pages leave open: the block's q and k are rotated at their absolute
 *               positions ctx_len[b] + i (Lmax when ctx_len is NULL) before their bf16
 *               rounding, interleaved pairs (2j, 2j+1) of each head turned by
 *               pos * rope_theta^(-2j/D); the cached context keys are taken as already rotated
 *               by the context tower. Negative or non-finite: TD_ERR_INVALID_ARG.
 *   paging      the context caches' layout (td_paging; page_table NULL: contiguous).
 *   h_out       NULL, or a device buffer, bf16 [B*S, d], 16-byte aligned, that receives the
 *               block's hidden state after the last layer: every row, the LM head's input
 *               (rows the step does not evaluate included). td_denoise_step only: a non-NULL
 *               h_out given to td_decode_block returns TD_ERR_INVALID_ARG (a loop has no
 *               single final state). Writing it changes no other output.
 *   attn_precision  a td_attn_precision for every attention of the step (anything else:
 *               TD_ERR_INVALID_ARG). */
typedef struct td_step_opts {
  int rule;
  float rope_theta;
  td_paging paging;
  void* h_out;
  int attn_precision;
} td_step_opts;

/* Selector for td_workspace_size(). */
enum {
  TD_FN_ADALN_MODULATE = 0,
  TD_FN_BLOCK_ATTENTION = 1,
  TD_FN_LMHEAD_COMMIT = 2,
  TD_FN_DENOISE_STEP = 3,
  TD_FN_DECODE_BLOCK = 4
};

/* Bytes of caller-provided scratch that entry point `fn` needs for `dims`; 0 if none,
 * (size_t)-1 if dims are invalid or unsupported. */
size_t td_workspace_size(const td_dims* dims, int fn);

/* Human-readable name of a status code (static storage, never NULL). */
const char* td_status_string(td_status s);

/* adaLN-single modulation ([chathome] inference paragraph: the diffusion timestep
 * modulates every layer through adaLN-single).
 *   m = E + phi (fp32 [6, d] each); for each row r of h:
 *   x_hat = (h_r - mean(h_r)) / sqrt(var(h_r) + eps)   (population variance, no affine)
 *   x_mod_r = bf16(x_hat * (1 + m[1]) + m[0])
 * h: bf16 [rows, d] (read only). x_mod: bf16 [rows, d] (written). No workspace.
 * Statistics in fp32. h and x_mod start on 16-byte boundaries; E and phi need only fp32
 * alignment (d % 256 == 0 with 16-byte aligned E and phi takes the vectorised kernel, any
 * other case a scalar one; both give the same result up to fp32 rounding).
 * Errors: TD_ERR_INVALID_ARG (null, rows <= 0, d <= 0, eps < 0, h or x_mod not 16-byte
 * aligned), TD_ERR_UNSUPPORTED (d % 8 != 0 or d > 8192). */
td_status td_adaln_modulate(const void* h, const float* E, const float* phi, int rows, int d,
                            float eps, void* x_mod, void* stream);

/* Fused block attention ([chathome] inference paragraph: bidirectional attention inside
 * the block, causal to past clean blocks, layer-aligned cross-attention to the context
 * tower's per-layer KV cache). For every sequence b, block position i, query head h,
 * with g = h / (Hq/Hkv) and L_b = ctx_len ? ctx_len[b] : Lmax:
 *   keys   = k_ctx[b, g, 0:L_b, :] followed by k_blk[b, 0:S, g, :]
 *   values = v_ctx[b, g, 0:L_b, :] followed by v_blk[b, 0:S, g, :]
 *   o[b, i, h, :] = bf16( sum_j softmax_j(q[b,i,h,:] . keys_j / sqrt(D)) values_j )
 * one softmax over the union (no mask: the cache holds only past tokens).
 *   q      bf16 [B, S, Hq, D]       k_blk, v_blk bf16 [B, S, Hkv, D]
 *   k_ctx, v_ctx bf16 [B, Hkv, Lmax, D]
 *   ctx_len int32 [B] or NULL (0 <= ctx_len[b] <= Lmax)
 *   paging  NULL (k_ctx, v_ctx contiguous as above) or a paged layout (td_paging: k_ctx,
 *           v_ctx are page pools)
 *   precision  a td_attn_precision (anything else: TD_ERR_INVALID_ARG)
 *   o      bf16 [B, S, Hq, D] (written)
 *   lse    fp32 [B, S, Hq] or NULL: natural log of sum_j exp(q . keys_j / sqrt(D))
 *   ws     >= td_workspace_size(dims, TD_FN_BLOCK_ATTENTION) bytes.
 * Only B, S, Hq, Hkv, D, Lmax of dims are read. */
td_status td_block_attention(const td_dims* dims, const void* q, const void* k_blk,
                             const void* v_blk, const void* k_ctx, const void* v_ctx,
                             const int* ctx_len, const td_paging* paging, int precision,
                             void* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/* LM head + confidence-masking commit ([chathome] generation and evaluation paragraphs:
 * tokens of the block commit when their confidence clears gamma; several commit per step).
 * For every row r = b*S + i:  z = h_r . W_lm^T (fp32 accumulate, never stored),
 *   conf[r] = max_v softmax(z)_v = 1 / sum_v exp(z_v - max z),
 *   pred[r] = the lowest v with z_v = max z.
 * Commit, per sequence b, rule TD_COMMIT_CONFIDENCE: C = { i : masked[b,i] && conf >= gamma };
 * if C is empty and some position is masked, C = { the lowest-index masked i of maximal
 * conf }. Rule TD_COMMIT_LEFT_TO_RIGHT: C = { the lowest-index masked i }. If force_all,
 * C = every masked i. For i in C: tokens[b,i] = pred, masked[b,i] = 0.
 * n_committed[b] = |C|; *all_done = 1 if no position of any sequence is still masked.
 *   h     bf16 [B*S, d]           w_lm bf16 [V, d]
 *   tokens int32 [B, S] in/out    masked uint8 [B, S] in/out (1 = still [MASK])
 *   conf  fp32 [B, S] out (every row)   pred int32 [B, S] out (every row)
 *   n_committed int32 [B] out           all_done int32 [1] out
 *   rule  a td_commit_rule (anything else: TD_ERR_INVALID_ARG)
 * Only B, S, d, V of dims are read. Committed positions are never rewritten. */
td_status td_lmhead_commit(const td_dims* dims, const void* h, const void* w_lm, float gamma,
                           int rule, int force_all, int* tokens, unsigned char* masked,
                           float* conf, int* pred, int* n_committed, int* all_done, void* ws,
                           size_t ws_bytes, void* stream);

/* One denoising step of the denoiser tower over the block ([chathome] inference and
 * generation paragraphs). If h is NULL the block's input is embedded from the tokens:
 *   h0[b, i] = bf16(emb[tokens[b, i]] + pos[i])   (emb bf16 [V+1, d], row V = [MASK];
 *   pos bf16 [S, d] stands in for the position information of the out-of-scope layers)
 * else h (bf16 [B*S, d], read only) is the input. Then for each layer l:
 *   m = E_l + phi_t; x_mod = adaLN(h) as in td_adaln_modulate (eps = 1e-6);
 *   [q | k | v] = bf16(x_mod . wqkv^T); o = td_block_attention(...);
 *   h = bf16(h + m[2] * (o . wo^T))            (m[2] is the gate)
 * (with opts->rope_theta > 0 the q and k of the block are rotated, see td_step_opts)
 * and finally td_lmhead_commit with opts->rule and force_all = (t == T), evaluated only
 * on the rows that can commit: those masked when the step starts, and under
 * TD_COMMIT_LEFT_TO_RIGHT before step T only the lowest masked row of each sequence
 * (committed rows need no logits; the last layer writes just those rows, compacted, and the
 * LM head reads their count on the device). Rows not evaluated get conf = 0 and pred = -1.
 *   phi_t fp32 [6, d]: the shared adaLN-single timestep vector of step t (1 <= t <= T).
 *   layers: HOST array of dims->n_layers td_layer structs (device pointers inside).
 *   ctx_len int32 [B] device or NULL.  Other outputs as in td_lmhead_commit.
 * Errors: TD_ERR_INVALID_ARG also when w_lm, or (on the embedding path) emb or pos, does
 * not start on a 16-byte boundary, or when a layer's weights, table or caches do not; h
 * may have any 2-byte alignment (it is copied into the workspace first). */
td_status td_denoise_step(const td_dims* dims, const td_layer* layers, const int* ctx_len,
                          const void* h, const void* emb, const void* pos, const void* w_lm,
                          const float* phi_t, int t, int T, float gamma,
                          const td_step_opts* opts, int* tokens, unsigned char* masked,
                          float* conf, int* pred, int* n_committed, int* all_done, void* ws,
                          size_t ws_bytes, void* stream);

/* Block decode loop ([chathome] generation paragraph: a block starts as S [MASK] tokens,
 * is refined for T steps and committed). Runs td_denoise_step (embedding path) for
 * t = t_start .. T with phi_t = phi_table[t-1] (fp32 [T, 6, d]) and stops after the first
 * step that leaves no position masked. tokens/masked hold the block state on entry
 * (all [MASK] for a fresh block; a partially committed state resumes a stopped loop).
 * steps_taken: HOST int, set to the number of steps run.
 * Execution: the steps t_start..T are captured once per distinct argument set into a CUDA
 * graph (on a stream private to the library) and replayed on `stream`, so the call
 * synchronises with the host once per block (plus one read of `masked` on entry). Each step
 * sits in a conditional graph node whose condition the previous step's commit sets to
 * "positions left": the steps after the one that committed the last position launch no
 * kernel. Where conditional nodes are not available the graph is one flat capture whose
 * kernels return at once when the previous step left nothing masked (see
 * td_decode_graph_form). If capture is not possible the steps run from a host loop that reads
 * all_done back after each step.
 * Returns TD_ERR_NOT_CONVERGED only if positions remain masked after step T (cannot
 * happen with force-commit at t == T; kept for callers that stop early). Alignment rules and
 * the other errors as in td_denoise_step (emb and pos are always read here). */
td_status td_decode_block(const td_dims* dims, const td_layer* layers, const int* ctx_len,
                          const void* emb, const void* pos, const void* w_lm,
                          const float* phi_table, int t_start, int T, float gamma,
                          const td_step_opts* opts, int* tokens, unsigned char* masked,
                          float* conf, int* pred, int* n_committed, int* all_done,
                          int* steps_taken, void* ws, size_t ws_bytes, void* stream);

/* The committed block's keys / values of one context-tower layer (the context tower's
 * forward pass itself is outside this library; its output is the input here).
 *   k, v  bf16 [B, S, Hkv, D] device, token-major */
typedef struct td_kv {
  const void* k;
  const void* v;
} td_kv;

/* Context-cache growth after a block commits ([chathome] generation paragraph: once a block
 * is committed the context tower takes it in, and the next block attends to it). For every
 * layer l, sequence b, block position i and KV head g:
 *   layers[l].k_ctx[b, g, ctx_len[b] + i, :] = block_kv[l].k[b, i, g, :]   (same for v)
 * then ctx_len[b] += S. The caches named by layers (k_ctx, v_ctx) are WRITTEN.
 *   block_kv: HOST array of dims->n_layers td_kv (device pointers inside).
 *   ctx_len  int32 [B] device, in/out.
 * A sequence whose cache would pass Lmax (or whose ctx_len is negative) is left unchanged
 * and the device error word reads ERR_CTX_FULL (0x600, see td_device_error).
 * With paging (non-NULL, page_table set) the caches are page pools and position pos of
 * sequence b is written to row pos % 128 of page page_table[b * max_pages + pos / 128]; the
 * caller maps the pages of the new positions before the call. A sequence whose new
 * positions map to a page-table entry outside [0, n_pages) is left unchanged as well (no row
 * written, ctx_len kept) and the device error word reads ERR_BAD_PAGE (0x700).
 * Only B, S, Hkv, D, Lmax, n_layers of dims are read. Errors: TD_ERR_INVALID_ARG (null or
 * misaligned pointers, Lmax < S, a malformed td_paging). Asynchronous on stream; no
 * workspace. */
td_status td_kv_append(const td_dims* dims, const td_layer* layers, const td_kv* block_kv,
                       int* ctx_len, const td_paging* paging, void* stream);

/* adaLN-single timestep map ([chathome] inference paragraph: the diffusion timestep modulates
 * every layer through adaLN-single, about 1.5 M parameters in all; the map from the timestep
 * to the shared vector is not given, and this is a reading of it): the table of shared
 * vectors phi(t), t = 1..T, that td_denoise_step and td_decode_block take:
 *   tau = t / T, s = 1000 tau, w_j = 10000^(-j/128), j = 0..127,
 *   e(tau) = [cos(s w_0) .. cos(s w_127), sin(s w_0) .. sin(s w_127)]   (256 values)
 *   phi_table[t-1, r, c] = (W_t e(tau) + b_t)[r*d + c]                   (r < 6, c < d)
 * computed in double precision and rounded to fp32 once.
 *   w_t fp32 [6*d, 256] device   b_t fp32 [6*d] device   phi_table fp32 [T, 6, d] device (out)
 * Errors: TD_ERR_INVALID_ARG (null pointer, d <= 0, T outside 1..65536), TD_ERR_UNSUPPORTED
 * (6*d > 2^30). Asynchronous on stream; no workspace. */
td_status td_timestep_table(const float* w_t, const float* b_t, int d, int T, float* phi_table,
                            void* stream);

/* Reads and clears the device error word that bounded waits write (0 = none); the
 * current device is used. Synchronises the device. Returns TD_ERR_DEVICE_TIMEOUT (with *code
 * set) when the word holds a wait code (0x100, 0x200 or 0x300), TD_ERR_CUDA if the read fails,
 * TD_OK otherwise.
 * Codes: 0x100 a TMA transfer, 0x200 an MMA, 0x300 a hand-off between warps did not complete
 * within the wait limit (about 2 s); 0x400 unusable TMEM; 0x500 a token id outside [0, V]
 * reached the embedding (it was read as [MASK]); 0x600 a cache append would pass Lmax;
 * 0x700 a page-table entry outside [0, n_pages). The first code recorded is kept. */
td_status td_device_error(int* code);

/* Diagnostic: launches one thread that waits, through the bounded wait all kernels use, on a
 * barrier that nothing completes, with a limit of limit_us microseconds (1 .. 2000000). The
 * wait gives up and records 0x300 in the device error word instead of hanging; a caller can
 * check that with td_device_error() (which also clears it) on its own GPU. No paper passage:
 * a property of this library. Asynchronous on stream. */
td_status td_check_bounded_wait(unsigned int limit_us, void* stream);

/* Diagnostic: the form of the decode-loop graphs (td_decode_block). form = 1 asks for the
 * chain of conditional nodes (the default), form = 2 for the flat capture, for graphs built
 * from now on in this process (each form is cached separately); any other value changes
 * nothing. Returns the form of the last graph built in this process (0 before the first).
 * No paper passage: a property of this library. No device work. */
int td_decode_graph_form(int form);

/* td_lmhead_commit without a caller-provided workspace. The pages have no counterpart: this
 * is a convenience of the library for callers that cannot allocate device memory, such as
 * a plugin running inside a host framework whose device memory is owned by that framework's
 * own pool or budget, or a latency-bound loop that must never call cudaMalloc / cudaFree
 * (both may synchronise the device). Same arguments, semantics and results as
 * td_lmhead_commit with rule TD_COMMIT_CONFIDENCE, minus rule, ws and ws_bytes.
 * Scratch: a fixed 16 MiB array in device memory that is part of this library, so every GPU
 * that loads the library holds it until the process exits. Its device address is looked up
 * on the first call made on each device (with that device current); make that first call
 * before any stream capture. The address is kept for the life of the process: after a
 * cudaDeviceReset() of that device it is stale, and this entry point must not be called on
 * that device again. Nothing is allocated, by this call or by that set-up.
 * Limit: 3 * align256(B*S * ceil(V / N_tile) * 4) + 256 bytes must fit in 16 MiB
 * (align256 rounds up to a multiple of 256; N_tile = 128 for B*S <= 128, 256 otherwise).
 * For example 2720 rows (B = 170, S = 16) at V = 131072 fit; larger problems return
 * TD_ERR_WORKSPACE with nothing launched.
 * All calls share the one array and it keeps the last call's contents (the commit counters
 * are cleared by every call): calls that can overlap on the GPU (different streams, or
 * different host threads) race on it and must be serialised by the caller. */
td_status td_lmhead_commit_static(const td_dims* dims, const void* h, const void* w_lm,
                                  float gamma, int force_all, int* tokens,
                                  unsigned char* masked, float* conf, int* pred,
                                  int* n_committed, int* all_done, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TD_H_ */
