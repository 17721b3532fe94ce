/*
 * li.h -- C ABI of libli_b300.so: the LatentIndex decode/prefill indexer scan
 * over a shared latent cache, for NVIDIA B300 (sm_103a).
 *
 * What the library computes (sources: "LatentIndex: Cross-Layer Sharing with
 * Layer-Specific Selection for Sparse Attention", summary page, Methodology,
 * eqs. (6)-(8) and the "Hierarchical Selection" paragraph; "LatentIndex --
 * Shared indexer cache, per-layer token choice", explainer page):
 *
 *   a group of G consecutive layers caches ONE latent c_t (r values) per
 *   token; layer l folds its decoder D_l (stored r x d) into each indexer-head
 *   query, q~_{l,h} = D_l q_{l,h}                                   (eq. 6)
 *   and scores every valid cached token with
 *   u_l(t) = sum_h w_{l,h} ReLU(q~_{l,h} . c_t + beta_{l,h})       (eq. 8)
 *   then keeps its own top-k token set.  Hierarchical selection (HS) lets the
 *   group's first layer (the anchor) propose its top-m candidates and the
 *   other layers (followers) rescore and select only inside them.
 *
 * Conventions (all entry points):
 *  - Pointers named as tensors are DEVICE pointers owned by the caller; the
 *    library never allocates device memory.  Tensors are dense, row-major, in
 *    the layout written next to each argument, with 16-byte aligned base
 *    addresses.  A NULL optional pointer means "absent" as documented.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call is asynchronous on that stream; its return value covers argument
 *    validation and launch errors only.  Errors a kernel detects on the device
 *    (a bounded wait that ran out) are latched in a per-device status word and
 *    read with li_device_status().
 *  - Argument errors are reported before any CUDA call is made.
 *  - Storage types: LI_F32 float, LI_BF16 bfloat16, LI_FP8_E4M3 OCP FP8 E4M3
 *    ("fn") codes with one fp32 scale per row: value = scale * decode(code).
 *    Scales must be >= 0 and finite.
 *  - Kernels are launched with programmatic stream serialization: a launch
 *    may be scheduled while the preceding kernel in the stream finishes.  The
 *    decode scans (li_score_group and li_native_score without q_pos, the HS
 *    anchor scan) issue the loads of their first cache tiles before waiting
 *    for that kernel.  A caller kernel that writes the latent / key cache and
 *    itself triggers programmatic dependents (griddepcontrol.launch_dependents)
 *    must do so only after those writes and a device-wide fence, as
 *    li_append_latent does; kernels launched without that trigger are waited
 *    for in full.
 *  - Calls are reentrant; concurrent calls on different streams are safe.
 *  - The library caches, per device, the device addresses of its own device
 *    variables (the status word; the scratch array of li_hs_select_noalloc),
 *    looked up on first use.  cudaDeviceReset() on a device invalidates them:
 *    do not call into the library on that device after a reset in the same
 *    process.
 */
#ifndef LI_B300_H
#define LI_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { LI_F32 = 0, LI_BF16 = 1, LI_FP8_E4M3 = 2 } li_dtype;

enum {
    LI_OK = 0,
    LI_ERR_INVALID_ARG = -1,   /* NULL required pointer, non-positive size, bad enum */
    LI_ERR_ALIGNMENT = -2,     /* a tensor base address is not 16-byte aligned        */
    LI_ERR_UNSUPPORTED = -3,   /* valid arguments outside what the kernels implement */
    LI_ERR_WORKSPACE = -4,     /* workspace missing or smaller than required         */
    LI_ERR_CUDA = -5,          /* a CUDA runtime/driver call or a launch failed      */
    LI_ERR_TIMEOUT = -6,       /* device: a bounded wait inside a kernel ran out     */
    LI_ERR_DEVICE_BOUNDS = -7  /* device: an index outside its tensor was skipped    */
};

/* Library version, major*10000 + minor*100 + patch. */
int li_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *li_status_string(int status);

/*
 * Query-side decoder absorption (summary page, eq. (6); explainer page:
 * q.(D c) = (D^T q).c lets the decoder act once on the query instead of on
 * every cached latent).
 *
 *   q      [B][T][G][H][d]  q_t in {LI_F32, LI_BF16}
 *   D      [G][r][d]        D_t in {LI_F32, LI_BF16}; NULL = identity
 *                           (requires r == d: rows of q are only converted /
 *                           quantised, which prepares native DSA queries)
 *   q_abs  [B][T][G][H][r]  out, abs_t in {LI_F32, LI_BF16, LI_FP8_E4M3}
 *   q_abs_scale [B][T][G][H] out fp32: required iff abs_t == LI_FP8_E4M3
 *                           (per-row scale = max|row| / 448), else ignored.
 * Accumulation is fp32; the result is rounded once to abs_t.
 * Limits: 1 <= d <= 1024, 1 <= r <= 256.
 */
int li_absorb_queries(const void *q, int q_t, const void *D, int D_t,
                      int B, int T, int G, int H, int d, int r,
                      void *q_abs, int abs_t, float *q_abs_scale, void *stream);

/*
 * Group scoring on the shared latent cache (summary page, eq. (8)), all G
 * layers of the group in one pass over the cache.
 *
 *   latent      [B][L][r]     lat_t; LI_FP8_E4M3 needs lat_scale [B][L];
 *                             lat_scale is optional (NULL = 1) otherwise
 *   q_abs       [B][T][G][H][r] abs_t, q_abs_scale [B][T][G][H] as produced
 *                             by li_absorb_queries (NULL = 1 unless fp8)
 *   w           [B][T][G][H]  fp32 head weights (query dependent)
 *   beta        [B][T][G][H]  fp32 or NULL (= 0): beta = q^N . b of eq. (6)
 *   q_pos       [T] int32 or NULL.  NULL: every cached token is valid (decode).
 *                             Otherwise query t sees tokens s <= q_pos[t]
 *                             (causal prefill); q_pos[t] >= 0.
 *   scores      [B][T][G][L]  fp32 out: u_l(t) for valid t.  Entries past a
 *                             query's causal limit are not written.
 * Supported dtype pairs: (F32, F32) on CUDA cores; (BF16, BF16) and
 * (FP8_E4M3, FP8_E4M3) on the tensor cores (tcgen05) when r % 64 == 0,
 * r <= 256 and H in {16, 32, 64, 128}: in one pass over the cache when
 * G*H <= 256, else in chunks of 256/H layers, one pass per chunk (G = 8 at
 * H = 64: two passes); any other pair or shape runs on CUDA cores when
 * G*H*r <= 8192 and r <= 256, else LI_ERR_UNSUPPORTED.
 */
int li_score_group(const void *latent, int lat_t, const float *lat_scale,
                   const void *q_abs, int abs_t, const float *q_abs_scale,
                   const float *w, const float *beta, const int32_t *q_pos,
                   int B, int T, int G, int H, int r, int L,
                   float *scores, void *stream);

/*
 * Workspace bytes li_topk can use for these sizes: non-zero when the rows are
 * longer than 32,768 scores and ceil(L / 32,768) * k <= 32,768 (for k = 2048,
 * L up to 524,288; for k = 8192, L up to 131,072).
 */
size_t li_topk_workspace_size(int64_t rows, int L, int k);

/*
 * Per-row top-k (summary page, TopK after eq. (8)): for each of `rows` score
 * rows of length L, the indices of the min(k, V) largest scores over the
 * valid prefix [0, V), V = valid_len[row] (NULL: V = L; values are clamped to
 * [0, L]).  Exact: a radix select on order-preserving 32-bit keys.  Among
 * equal scores at the threshold the lower index is taken.  NaN scores are
 * not allowed.
 *
 *   scores [rows][L] fp32; idx [rows][k] int32 out (set in unspecified order,
 *   slots past min(k, V) hold -1); vals [rows][k] fp32 out or NULL (the score
 *   of each selected index, -inf in padded slots).
 *   ws     optional device workspace (16-byte aligned) of ws_bytes; with at
 *          least li_topk_workspace_size(rows, L, k) bytes, rows longer than
 *          32,768 and valid_len == NULL are selected in two passes (the exact
 *          top-k of each 32,768-score segment, then of the segments'
 *          candidates, ties by position) with more parallelism.  The result
 *          is the same with or without it; NULL / too small = one pass.
 *          Few rows (ceil(L / 8,192) * rows at most the SM count, L <=
 *          131,072) are instead each spread over a thread-block cluster,
 *          with or without ws.
 * Limits: 1 <= k <= 2^30, L < 2^31.
 */
int li_topk(const float *scores, int64_t rows, int L, const int32_t *valid_len, int k,
            int32_t *idx, float *vals, void *ws, size_t ws_bytes, void *stream);

/* Workspace bytes li_hs_select needs for these sizes. */
size_t li_hs_workspace_size(int B, int G, int L, int m, int k);

/*
 * Hierarchical selection for one decode step of B sequences (summary page,
 * "Hierarchical Selection"; explainer page: the anchor fills a cart of
 * candidates and each follower picks its own top-k from the cart only).
 *
 * The anchor (layer 0 of the group) scores all L cached tokens and keeps its
 * top-m positions as the candidate set C_b (m >= k) and its top-k as its own
 * selection; every follower l = 1..G-1 rescores only the min(m, L) candidate
 * rows of the latent and keeps its top-k inside C_b.  Scored positions per
 * sequence: L + (G-1) min(m, L).
 *
 *   latent, lat_t, lat_scale, q_abs (T = 1), abs_t, q_abs_scale, w, beta
 *                    as for li_score_group with T = 1
 *   cand [B][m] int32 out: anchor candidates (-1 padded when L < m)
 *   idx  [B][G][k] int32 out: per-layer selections (-1 padded)
 *   ws   device workspace of at least li_hs_workspace_size(B, G, L, m, k)
 *        bytes, 256-byte aligned.
 * Ties at a threshold go to the lower token position (followers: for
 * m <= 32,768; beyond that to the earlier slot of the candidate list).
 */
int li_hs_select(const void *latent, int lat_t, const float *lat_scale,
                 const void *q_abs, int abs_t, const float *q_abs_scale,
                 const float *w, const float *beta,
                 int B, int G, int H, int r, int L, int m, int k,
                 int32_t *cand, int32_t *idx, void *ws, size_t ws_bytes, void *stream);

/*
 * li_hs_select with per-launch timing (a diagnostic entry point; the pages
 * have no counterpart).  Same arguments, work and results as li_hs_select,
 * plus `events`: five caller-created cudaEvent_t handles.  events[i] is
 * recorded on `stream` before launch i of the selection and events[4] after
 * the last one: 0 anchor scan, 1 anchor top-m (candidates and their anchor
 * scores), 2 follower rescoring of the candidates (empty interval when
 * G = 1), 3 the top-k of every layer inside the candidates (one launch).
 * Recording an event between two launches ends their programmatic launch
 * overlap, so the intervals add up to a little more than an unprofiled call.
 * LI_ERR_INVALID_ARG when events is NULL.
 */
int li_hs_select_profiled(const void *latent, int lat_t, const float *lat_scale,
                          const void *q_abs, int abs_t, const float *q_abs_scale,
                          const float *w, const float *beta,
                          int B, int G, int H, int r, int L, int m, int k,
                          int32_t *cand, int32_t *idx, void *ws, size_t ws_bytes,
                          void *const *events, void *stream);

/*
 * Hierarchical selection without a caller workspace.  The paper has no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory where they run the indexer -- for example a plugin inside a serving
 * engine whose device memory is all owned by the engine's pool, or a decode
 * loop that must not call cudaMalloc (it can synchronise the device).
 *
 * Same arguments, outputs and results as li_hs_select, minus ws / ws_bytes.
 * The scratch is a fixed 8 MiB device array inside this library (8,388,608
 * bytes; every GPU that loads the library holds it until the process exits).
 * Sizes whose li_hs_workspace_size(B, G, L, m, k) exceeds 8 MiB are rejected
 * with LI_ERR_WORKSPACE before anything runs (B = 8, L = 131072, m = 8192,
 * G = 4 needs 7 MiB).  The call allocates nothing.
 *  - The first call on a device, made with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress) and caches it; make that
 *    first call before any stream capture.
 *  - All calls on a device share the one array and leave their contents in
 *    it; nothing in it has to start at zero (every value a call reads was
 *    written earlier in the same call).  Calls that may overlap on the GPU
 *    (different streams without ordering between them) race on the array:
 *    order them, or use li_hs_select with separate workspaces.
 */
int li_hs_select_noalloc(const void *latent, int lat_t, const float *lat_scale,
                         const void *q_abs, int abs_t, const float *q_abs_scale,
                         const float *w, const float *beta,
                         int B, int G, int H, int r, int L, int m, int k,
                         int32_t *cand, int32_t *idx, void *stream);

/*
 * Native per-layer DSA lightning indexer over one layer's own key cache, the
 * baseline LatentIndex replaces (explainer page: "DSA lightning indexer",
 * "Indexer key cache" of 132 B per token per layer = 128 fp8 values + one
 * fp32 scale):  I_t = sum_h w_h ReLU(q_h . k_t).
 *
 *   keys  [B][L][d]  key_t (LI_FP8_E4M3 with key_scale [B][L], or LI_BF16)
 *   q     [B][H][d]  q_t matching key_t (fp8 rows need q_scale [B][H]; use
 *                    li_absorb_queries with D = NULL to prepare them)
 *   w     [B][H]     fp32
 *   scores [B][L]    fp32 out
 * Same kernels and limits as li_score_group with G = 1, T = 1, r = d.
 */
int li_native_score(const void *keys, int key_t, const float *key_scale,
                    const void *q, int q_t, const float *q_scale, const float *w,
                    int B, int H, int d, int L, float *scores, void *stream);

/*
 * Latent-cache append (summary page, Methodology, "Shared Latent Cache",
 * eqs. (1)-(2)): for one new token per sequence, the shared latent
 *     c = [Q_t P_R^T x ; P_N^T x]
 * of the anchor layer's hidden state x, written into the cache at the
 * token's position.  Q_t rotates the RoPE branch as complex pairs
 * (c_2i, c_2i+1) by the angle t * rope_base^(-2i/rR).
 *
 *   x         [B][dm]  x_t in {LI_F32, LI_BF16}
 *   P         [r][dm]  P_t in {LI_F32, LI_BF16}; rows 0 .. rR-1 are P_R^T,
 *                      rows rR .. r-1 are P_N^T
 *   pos       [B] int32: position t of the token (rotation angle) and the
 *                      cache row it is written to
 *   latent    [B][L][r] lat_t in {LI_F32, LI_BF16, LI_FP8_E4M3}: row pos[b]
 *                      of sequence b is written, nothing else
 *   lat_scale [B][L] fp32: required for LI_FP8_E4M3 (the row's scale
 *                      max|c| / 448 is written at pos[b]), ignored otherwise
 * fp32 accumulation; fp8 codes rounded to nearest even, saturating.
 * A position outside [0, L) writes nothing and latches LI_ERR_DEVICE_BOUNDS.
 * Limits: 1 <= r <= 256, 0 <= rR <= r with rR even, 1 <= dm <= 2^24,
 * rope_base > 0.
 */
int li_append_latent(const void *x, int x_t, const void *P, int P_t, const int32_t *pos,
                     int B, int dm, int r, int rR, float rope_base,
                     void *latent, int lat_t, float *lat_scale, int L, void *stream);

/*
 * Test hook for the device-side watchdog (no counterpart on the pages).
 * Launches one CTA that allocates tensor memory and waits, with the bounded
 * mbarrier wait every kernel of this library uses, on a barrier that nothing
 * ever arrives on.  After `limit_us` microseconds (1 ... 1,000,000) the wait
 * gives up and latches LI_ERR_TIMEOUT in the device status word; the CTA
 * frees its tensor memory and exits, leaving the context usable.  The next
 * li_device_status() returns LI_ERR_TIMEOUT.  Returns LI_ERR_INVALID_ARG for
 * a limit out of range, LI_ERR_CUDA if the launch fails.
 */
int li_selftest_wait_timeout(unsigned int limit_us, void *stream);

/*
 * Synchronises `stream`, then returns and clears the calling device's status
 * word: LI_OK, or the first device-side error latched since the last call
 * (LI_ERR_TIMEOUT, LI_ERR_DEVICE_BOUNDS), or LI_ERR_CUDA if the
 * synchronisation itself failed.
 */
int li_device_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LI_B300_H */
