// li_api.cu -- the C ABI of libli_b300.so (declared in include/li.h).
//
// Each entry point validates its arguments on the host (returning a status
// before any CUDA call when they are wrong), picks the kernel for the dtype
// pair and shape, and launches asynchronously on the caller's stream.  The
// library owns no device memory except one status word per device, where
// kernels latch device-side errors (a bounded wait that ran out, an index
// outside its tensor); li_device_status() reads and clears it.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>

#include "li_internal.cuh"

namespace li {

__device__ int g_li_status;

int *device_status_ptr()
{
    constexpr int kMaxDev = 64;
    static std::atomic<int *> cache[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return nullptr;
    int *p = cache[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_li_status) != cudaSuccess)
            return nullptr;
        p = static_cast<int *>(addr);
        cache[dev].store(p, std::memory_order_release);
    }
    return p;
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype(int t) { return t == LI_F32 || t == LI_BF16 || t == LI_FP8_E4M3; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Two-pass selection of long rows: pass 1 takes the exact top-k of every
// kTopkRegRow-score segment (candidates carry their position in the whole
// row; unused slots hold position INT32_MAX and -inf), pass 2 the top-k of a
// row's segment candidates, ties broken through the candidates' positions.
// The global top-k is inside the union of the segments' top-k (fewer than k
// scores of the row beat any member, so fewer than k of its segment do), so
// the result equals a one-pass selection.  Used for rows without a valid
// length whose segment candidates fit one register-resident row.
int64_t topk_segments(int L, int k)
{
    if (L <= kTopkRegRow || k <= 0 || k > kTopkRegRow)
        return 0;
    const int64_t S = (static_cast<int64_t>(L) + kTopkRegRow - 1) / kTopkRegRow;
    return S * k <= kTopkRegRow ? S : 0;
}

size_t topk_two_pass_bytes(int64_t rows, int L, int k)
{
    const int64_t S = topk_segments(L, k);
    if (rows <= 0 || S == 0)
        return 0;
    return 2 * align256(sizeof(float) * static_cast<size_t>(rows * S * k));
}

// p: the one-pass parameters (rows_per_group == 1, no map, no valid_len).
cudaError_t launch_topk_two_pass(const TopkParams &p, void *ws, cudaStream_t s)
{
    const int64_t S = topk_segments(p.L_row, p.k);
    const size_t n = static_cast<size_t>(p.rows * S * p.k);
    float *cv = static_cast<float *>(ws);
    int32_t *ci = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) + align256(sizeof(float) * n));
    TopkParams a = p;
    a.rows = p.rows * S;
    a.idx = ci;
    a.vals = cv;
    a.vals_stride = 0;
    a.rows_per_group = 1;
    a.group_stride = 1;
    a.row_offset = 0;
    a.segs = static_cast<int>(S);
    a.seg_len = kTopkRegRow;
    a.pad_idx = INT32_MAX;
    cudaError_t e = launch_topk(a, s);
    if (e != cudaSuccess)
        return e;
    TopkParams b = p;
    b.scores = cv;
    b.in_stride = S * p.k;
    b.L_row = static_cast<int>(S * p.k);
    b.map = ci;
    b.map_stride = S * p.k;
    return launch_topk(b, s);
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? LI_OK : LI_ERR_CUDA; }

// Shared memory the CUDA-core scorer needs for this shape.
size_t simt_smem(int Gs, int H, int r)
{
    const size_t N = static_cast<size_t>(Gs) * H;
    return sizeof(float) * (N * r + 2 * N + 128 * (static_cast<size_t>(r) + 1));
}

// Validates the scoring arguments shared by li_score_group / li_native_score /
// li_hs_select.  Returns LI_OK or an error status.
int check_score_args(const void *latent, int lat_t, const float *lat_scale, const void *q_abs,
                     int abs_t, const float *q_abs_scale, const float *w, const float *beta,
                     const int32_t *q_pos, const void *out, int B, int T, int G, int H, int r, int L)
{
    if (!latent || !q_abs || !w || !out)
        return LI_ERR_INVALID_ARG;
    if (!valid_dtype(lat_t) || !valid_dtype(abs_t))
        return LI_ERR_INVALID_ARG;
    if (B <= 0 || T <= 0 || G <= 0 || H <= 0 || r <= 0 || L <= 0)
        return LI_ERR_INVALID_ARG;
    if (lat_t == LI_FP8_E4M3 && !lat_scale)
        return LI_ERR_INVALID_ARG;
    if (abs_t == LI_FP8_E4M3 && !q_abs_scale)
        return LI_ERR_INVALID_ARG;
    if (!aligned16(latent) || !aligned16(q_abs) || !aligned16(w) || !aligned16(out) ||
        !aligned16(lat_scale) || !aligned16(q_abs_scale) || !aligned16(beta) || !aligned16(q_pos))
        return LI_ERR_ALIGNMENT;
    if (r > 256)
        return LI_ERR_UNSUPPORTED;
    return LI_OK;
}

// More layers than one tensor-core tile holds (Gs * H > 256): the layers are
// scored in chunks of 256 / H, one pass over the cache per chunk, each chunk
// writing its own rows of the score tensor.  Returns the layers per chunk, or
// 0 when the chunks are not tensor-core shapes.
int tc_chunk_layers(const ScoreParams &p)
{
    if (p.Gs <= 1 || p.H <= 0 || p.H > 256)
        return 0;
    ScoreParams q = p;
    q.Gs = 256 / p.H;
    return q.Gs >= 1 && q.Gs < p.Gs && score_tc_supported(q) ? q.Gs : 0;
}

int run_score(const ScoreParams &p, cudaStream_t s)
{
    if (score_tc_supported(p))
        return cuda_status(launch_score_tc(p, s));
    if (const int gc = tc_chunk_layers(p)) {
        for (int c = 0; c < p.Gs; c += gc) {
            ScoreParams q = p;
            q.Gout = p.Gout ? p.Gout : p.Gs;
            q.gout0 = p.gout0 + c;
            q.g0 = p.g0 + c;
            q.Gs = p.Gs - c < gc ? p.Gs - c : gc;
            const int st = cuda_status(score_tc_supported(q) ? launch_score_tc(q, s)
                                                             : launch_score_simt(q, s));
            if (st != LI_OK)
                return st;
        }
        return LI_OK;
    }
    if (simt_smem(p.Gs, p.H, p.r) <= 227 * 1024)
        return cuda_status(launch_score_simt(p, s));
    return LI_ERR_UNSUPPORTED;
}

bool score_supported(const ScoreParams &p)
{
    return score_tc_supported(p) || tc_chunk_layers(p) > 0 || simt_smem(p.Gs, p.H, p.r) <= 227 * 1024;
}

} // namespace
} // namespace li

using namespace li;

extern "C" {

int li_version(void) { return 100; }

const char *li_status_string(int status)
{
    switch (status) {
    case LI_OK: return "LI_OK";
    case LI_ERR_INVALID_ARG: return "LI_ERR_INVALID_ARG: invalid argument";
    case LI_ERR_ALIGNMENT: return "LI_ERR_ALIGNMENT: tensor base address not 16-byte aligned";
    case LI_ERR_UNSUPPORTED: return "LI_ERR_UNSUPPORTED: dtype pair or shape not implemented";
    case LI_ERR_WORKSPACE: return "LI_ERR_WORKSPACE: workspace missing or too small";
    case LI_ERR_CUDA: return "LI_ERR_CUDA: CUDA call or launch failed";
    case LI_ERR_TIMEOUT: return "LI_ERR_TIMEOUT: a bounded wait inside a kernel ran out";
    case LI_ERR_DEVICE_BOUNDS: return "LI_ERR_DEVICE_BOUNDS: an index outside its tensor was skipped";
    default: return "unknown status";
    }
}

int li_absorb_queries(const void *q, int q_t, const void *D, int D_t, int B, int T, int G, int H,
                      int d, int r, void *q_abs, int abs_t, float *q_abs_scale, void *stream)
{
    if (!q || !q_abs)
        return LI_ERR_INVALID_ARG;
    if ((q_t != LI_F32 && q_t != LI_BF16) || !valid_dtype(abs_t))
        return LI_ERR_INVALID_ARG;
    if (D && D_t != LI_F32 && D_t != LI_BF16)
        return LI_ERR_INVALID_ARG;
    if (B <= 0 || T <= 0 || G <= 0 || H <= 0 || d <= 0 || r <= 0)
        return LI_ERR_INVALID_ARG;
    if (!D && r != d)
        return LI_ERR_INVALID_ARG;
    if (abs_t == LI_FP8_E4M3 && !q_abs_scale)
        return LI_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(D) || !aligned16(q_abs) ||
        (abs_t == LI_FP8_E4M3 && !aligned16(q_abs_scale)))
        return LI_ERR_ALIGNMENT;
    if (r > 256 || d > 1024 || G > 65535)
        return LI_ERR_UNSUPPORTED;
    const int64_t N = static_cast<int64_t>(B) * T;
    if (N * H > 0x7FFFFFFFll * 64)
        return LI_ERR_UNSUPPORTED;
    AbsorbParams p;
    p.q = q;
    p.D = D;
    p.q_abs = q_abs;
    p.q_abs_scale = abs_t == LI_FP8_E4M3 ? q_abs_scale : nullptr;
    p.q_t = q_t;
    p.D_t = D ? D_t : LI_F32;
    p.abs_t = abs_t;
    p.N = static_cast<int>(N);
    p.G = G;
    p.H = H;
    p.d = d;
    p.r = r;
    if (N > 0x7FFFFFFF)
        return LI_ERR_UNSUPPORTED;
    return cuda_status(launch_absorb(p, static_cast<cudaStream_t>(stream)));
}

int li_score_group(const void *latent, int lat_t, const float *lat_scale, const void *q_abs,
                   int abs_t, const float *q_abs_scale, const float *w, const float *beta,
                   const int32_t *q_pos, int B, int T, int G, int H, int r, int L, float *scores,
                   void *stream)
{
    int st = check_score_args(latent, lat_t, lat_scale, q_abs, abs_t, q_abs_scale, w, beta, q_pos,
                              scores, B, T, G, H, r, L);
    if (st != LI_OK)
        return st;
    ScoreParams p{};
    p.latent = latent;
    p.lat_scale = lat_scale;
    p.q_abs = q_abs;
    p.q_abs_scale = q_abs_scale;
    p.w = w;
    p.beta = beta;
    p.q_pos = q_pos;
    p.gather_idx = nullptr;
    p.scores = scores;
    p.lat_t = lat_t;
    p.abs_t = abs_t;
    p.B = B;
    p.T = T;
    p.Gtot = G;
    p.g0 = 0;
    p.Gs = G;
    p.H = H;
    p.r = r;
    p.L_lat = L;
    p.L_out = L;
    p.n_gather = 0;
    if (!score_supported(p))
        return LI_ERR_UNSUPPORTED;
    p.status = device_status_ptr();
    if (!p.status)
        return LI_ERR_CUDA;
    return run_score(p, static_cast<cudaStream_t>(stream));
}

size_t li_topk_workspace_size(int64_t rows, int L, int k)
{
    return topk_two_pass_bytes(rows, L, k);
}

int li_topk(const float *scores, int64_t rows, int L, const int32_t *valid_len, int k, int32_t *idx,
            float *vals, void *ws, size_t ws_bytes, void *stream)
{
    if (!scores || !idx)
        return LI_ERR_INVALID_ARG;
    if (rows < 0 || L < 0 || k <= 0 || k > (1 << 30))
        return LI_ERR_INVALID_ARG;
    if (!aligned16(scores) || !aligned16(idx) || !aligned16(vals) || !aligned16(valid_len) ||
        !aligned16(ws))
        return LI_ERR_ALIGNMENT;
    if (rows == 0)
        return LI_OK;
    TopkParams p{};
    p.scores = scores;
    p.rows = rows;
    p.in_stride = L;
    p.L_row = L;
    p.valid_len = valid_len;
    p.k = k;
    p.idx = idx;
    p.vals = vals;
    p.rows_per_group = 1;
    p.group_stride = 1;
    p.row_offset = 0;
    p.map = nullptr;
    p.map_stride = 0;
    p.status = device_status_ptr();
    if (!p.status)
        return LI_ERR_CUDA;
    const size_t two = topk_two_pass_bytes(rows, L, k);
    if (ws && two > 0 && ws_bytes >= two && !valid_len && !topk_cluster_path(p))
        return cuda_status(launch_topk_two_pass(p, ws, static_cast<cudaStream_t>(stream)));
    return cuda_status(launch_topk(p, static_cast<cudaStream_t>(stream)));
}

size_t li_hs_workspace_size(int B, int G, int L, int m, int k)
{
    if (B <= 0 || G <= 0 || L <= 0 || m <= 0 || k <= 0)
        return 0;
    const size_t anchor = align256(sizeof(float) * static_cast<size_t>(B) * L);
    const size_t cand_scores = align256(sizeof(float) * static_cast<size_t>(B) * G * m);
    return anchor + cand_scores + topk_two_pass_bytes(B, L, m);
}

} // extern "C"

namespace li {

int hs_check_args(const void *latent, int lat_t, const float *lat_scale, const void *q_abs,
                  int abs_t, const float *q_abs_scale, const float *w, const float *beta, int B,
                  int G, int H, int r, int L, int m, int k, const int32_t *cand, const int32_t *idx)
{
    const int st = check_score_args(latent, lat_t, lat_scale, q_abs, abs_t, q_abs_scale, w, beta,
                                    nullptr, cand, B, 1, G, H, r, L);
    if (st != LI_OK)
        return st;
    if (!idx || m <= 0 || k <= 0 || m < k)
        return LI_ERR_INVALID_ARG;
    if (!aligned16(idx))
        return LI_ERR_ALIGNMENT;
    return LI_OK;
}

namespace {

// The four launches of hierarchical selection (anchor scan, anchor top-m,
// follower rescoring, every layer's top-k inside the candidates); when `ev`
// is given, ev[i] is recorded on the stream before launch i and ev[4] after
// the last one.
int hs_select_impl(const void *latent, int lat_t, const float *lat_scale, const void *q_abs,
                   int abs_t, const float *q_abs_scale, const float *w, const float *beta, int B,
                   int G, int H, int r, int L, int m, int k, int32_t *cand, int32_t *idx, void *ws,
                   size_t ws_bytes, void *stream, cudaEvent_t const *ev)
{
    int st = hs_check_args(latent, lat_t, lat_scale, q_abs, abs_t, q_abs_scale, w, beta, B, G, H, r,
                           L, m, k, cand, idx);
    if (st != LI_OK)
        return st;
    const size_t need = li_hs_workspace_size(B, G, L, m, k);
    if (!ws || ws_bytes < need)
        return LI_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return LI_ERR_ALIGNMENT;

    // workspace: anchor scores [B][L], then the candidates' scores of every
    // layer [B][G][m] (row 0 the anchor's, from the top-m pass; rows 1..G-1
    // the followers' rescoring), then the top-m pass's own scratch
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    float *anchor = reinterpret_cast<float *>(wsb);
    float *cs = reinterpret_cast<float *>(wsb + align256(sizeof(float) * static_cast<size_t>(B) * L));
    void *tws = reinterpret_cast<uint8_t *>(cs) +
                align256(sizeof(float) * static_cast<size_t>(B) * G * m);
    const int nc = m < L ? m : L;

    ScoreParams a{};
    a.latent = latent;
    a.lat_scale = lat_scale;
    a.q_abs = q_abs;
    a.q_abs_scale = q_abs_scale;
    a.w = w;
    a.beta = beta;
    a.q_pos = nullptr;
    a.gather_idx = nullptr;
    a.scores = anchor;
    a.lat_t = lat_t;
    a.abs_t = abs_t;
    a.B = B;
    a.T = 1;
    a.Gtot = G;
    a.g0 = 0;
    a.Gs = 1;
    a.H = H;
    a.r = r;
    a.L_lat = L;
    a.L_out = L;
    a.n_gather = 0;
    ScoreParams f = a;
    f.gather_idx = cand;
    f.scores = cs;
    f.g0 = 1;
    f.Gs = G - 1;
    f.L_out = m;
    f.n_gather = nc;
    f.Gout = G;          // rows 1..G-1 of each sequence's [G][m] block
    f.gout0 = 1;
    if (!score_supported(a) || (G > 1 && !score_supported(f)))
        return LI_ERR_UNSUPPORTED;

    int *status = device_status_ptr();
    if (!status)
        return LI_ERR_CUDA;
    a.status = f.status = status;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    auto mark = [&](int i) {
        if (ev != nullptr && ev[i] != nullptr)
            cudaEventRecord(ev[i], s);
    };
    // 1. anchor scores over all L positions
    mark(0);
    st = run_score(a, s);
    if (st != LI_OK)
        return st;
    // 2. anchor top-m -> candidate set, its scores into row 0 of [B][G][m]
    mark(1);
    TopkParams t{};
    t.scores = anchor;
    t.rows = B;
    t.in_stride = L;
    t.L_row = L;
    t.valid_len = nullptr;
    t.k = m;
    t.idx = cand;
    t.vals = cs;
    t.vals_stride = static_cast<int64_t>(G) * m;
    t.rows_per_group = 1;
    t.group_stride = 1;
    t.row_offset = 0;
    t.map = nullptr;
    t.map_stride = 0;
    t.status = status;
    st = cuda_status(topk_two_pass_bytes(B, L, m) > 0 && !topk_cluster_path(t)
                         ? launch_topk_two_pass(t, tws, s)
                         : launch_topk(t, s));
    if (st != LI_OK)
        return st;
    // 3. followers rescore the candidate rows of the latent (rows 1..G-1)
    mark(2);
    if (G > 1) {
        st = run_score(f, s);
        if (st != LI_OK)
            return st;
    }
    // 4. every layer's top-k inside the candidates, one launch over B x G rows
    mark(3);
    TopkParams tk = t;
    tk.scores = cs;
    tk.rows = static_cast<int64_t>(B) * G;
    tk.in_stride = m;
    tk.L_row = nc;
    tk.k = k;
    tk.idx = idx;
    tk.vals = nullptr;
    tk.vals_stride = 0;
    tk.rows_per_group = G;
    tk.group_stride = G;
    tk.row_offset = 0;
    tk.map = cand;
    tk.map_stride = m;
    st = cuda_status(launch_topk(tk, s));
    mark(4);
    return st;
}

} // namespace
} // namespace li

extern "C" {

int li_hs_select(const void *latent, int lat_t, const float *lat_scale, const void *q_abs, int abs_t,
                 const float *q_abs_scale, const float *w, const float *beta, int B, int G, int H,
                 int r, int L, int m, int k, int32_t *cand, int32_t *idx, void *ws, size_t ws_bytes,
                 void *stream)
{
    return hs_select_impl(latent, lat_t, lat_scale, q_abs, abs_t, q_abs_scale, w, beta, B, G, H, r,
                          L, m, k, cand, idx, ws, ws_bytes, stream, nullptr);
}

int li_hs_select_profiled(const void *latent, int lat_t, const float *lat_scale, const void *q_abs,
                          int abs_t, const float *q_abs_scale, const float *w, const float *beta,
                          int B, int G, int H, int r, int L, int m, int k, int32_t *cand,
                          int32_t *idx, void *ws, size_t ws_bytes, void *const *events,
                          void *stream)
{
    if (!events)
        return LI_ERR_INVALID_ARG;
    cudaEvent_t ev[5];
    for (int i = 0; i < 5; ++i)
        ev[i] = static_cast<cudaEvent_t>(events[i]);
    return hs_select_impl(latent, lat_t, lat_scale, q_abs, abs_t, q_abs_scale, w, beta, B, G, H, r,
                          L, m, k, cand, idx, ws, ws_bytes, stream, ev);
}

int li_native_score(const void *keys, int key_t, const float *key_scale, const void *q, int q_t,
                    const float *q_scale, const float *w, int B, int H, int d, int L, float *scores,
                    void *stream)
{
    return li_score_group(keys, key_t, key_scale, q, q_t, q_scale, w, nullptr, nullptr, B, 1, 1, H,
                          d, L, scores, stream);
}

int li_append_latent(const void *x, int x_t, const void *P, int P_t, const int32_t *pos, int B,
                     int dm, int r, int rR, float rope_base, void *latent, int lat_t, float *lat_scale,
                     int L, void *stream)
{
    if (!x || !P || !pos || !latent || B < 0 || dm < 1 || dm > (1 << 24) || r < 1 || r > 256 ||
        rR < 0 || rR > r || (rR & 1) || L < 1 || !(rope_base > 0.f))
        return LI_ERR_INVALID_ARG;
    if ((x_t != LI_F32 && x_t != LI_BF16) || (P_t != LI_F32 && P_t != LI_BF16) ||
        (lat_t != LI_F32 && lat_t != LI_BF16 && lat_t != LI_FP8_E4M3))
        return LI_ERR_INVALID_ARG;
    if (lat_t == LI_FP8_E4M3 && !lat_scale)
        return LI_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(P) || !aligned16(pos) || !aligned16(latent) || !aligned16(lat_scale))
        return LI_ERR_ALIGNMENT;
    if (B == 0)
        return LI_OK;
    AppendParams a{};
    a.x = x;
    a.P = P;
    a.pos = pos;
    a.latent = latent;
    a.lat_scale = lat_scale;
    a.x_t = x_t;
    a.P_t = P_t;
    a.lat_t = lat_t;
    a.B = B;
    a.dm = dm;
    a.r = r;
    a.rR = rR;
    a.L = L;
    a.base = rope_base;
    a.vec = dm % 8 == 0;
    a.status = device_status_ptr();
    if (!a.status)
        return LI_ERR_CUDA;
    return cuda_status(launch_append(a, static_cast<cudaStream_t>(stream)));
}

int li_device_status(void *stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LI_ERR_CUDA;
    int *p = device_status_ptr();
    if (!p)
        return LI_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return LI_ERR_CUDA;
    if (v != 0 && cudaMemset(p, 0, sizeof v) != cudaSuccess)
        return LI_ERR_CUDA;
    return v;
}

} // extern "C"
