// li_internal.cuh -- kernel parameter blocks and launchers shared by the
// library's translation units (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda.h>           // CUtensorMap and the tensor-map encoder's types
#include <cuda_runtime.h>

#include "../../include/li.h"

namespace li {

// cuTensorMapEncodeTiled from the driver (looked up once), or nullptr.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();
// Multiprocessors of the current device (cached per device).
int sm_count();

// Upper bound for any single mbarrier wait inside a kernel (ns).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// ------------------------------------------------------------- absorption
struct AbsorbParams {
    const void *q;        // [N][G][H][d]
    const void *D;        // [G][r][d] or nullptr (identity)
    void *q_abs;          // [N][G][H][r]
    float *q_abs_scale;   // [N][G][H] (fp8 only)
    int q_t, D_t, abs_t;
    int N, G, H, d, r;
};
cudaError_t launch_absorb(const AbsorbParams &p, cudaStream_t s);
// Tensor-core absorption (bf16 q and D, 64 | d <= 256, 32 | r <= 256,
// H in {16, 32, 64, 128}); launch_absorb uses it when it applies.
bool absorb_tc_supported(const AbsorbParams &p);
cudaError_t launch_absorb_tc(const AbsorbParams &p, cudaStream_t s);

// ------------------------------------------------------------- latent append
struct AppendParams {
    const void *x;         // [B][dm] anchor hidden state of the new token
    const void *P;         // [r][dm]: rows < rR are P_R^T, the rest P_N^T
    const int32_t *pos;    // [B] token position (rotary angle and cache row)
    void *latent;          // [B][L][r]
    float *lat_scale;      // [B][L] (fp8 caches)
    int *status;
    int x_t, P_t, lat_t;
    int B, dm, r, rR, L;
    float base;            // rotary base
    bool vec;              // dm % 8 == 0 and 16-byte aligned rows: vector loads
    int kc = 0;            // hidden elements per CTA of a cluster (set by launch_append)
    int kw = 0;            // hidden elements of P staged in shared memory at a time
    double theta[128];     // rotary frequencies base^(-2i / rR) (set by launch_append)
};
constexpr int kMaxRopePairs = 128;
cudaError_t launch_append(const AppendParams &p, cudaStream_t s);

// ------------------------------------------------------------- scoring
// One scoring launch evaluates eq. (8) for a contiguous range of Gs layers
// [g0, g0 + Gs) of a group of Gtot layers, either over every cached token
// (scan mode) or over a per-sequence list of gathered token indices.
struct ScoreParams {
    const void *latent;          // [B][L_lat][r]
    const float *lat_scale;      // [B][L_lat] or nullptr
    const void *q_abs;           // [B][T][Gtot][H][r]
    const float *q_abs_scale;    // [B][T][Gtot][H] or nullptr
    const float *w;              // [B][T][Gtot][H]
    const float *beta;           // [B][T][Gtot][H] or nullptr
    const int32_t *q_pos;        // [T] or nullptr (scan mode only)
    const int32_t *gather_idx;   // [B][L_out] or nullptr (gather mode)
    float *scores;               // [B][T][Gout][L_out]: layer l of the launch -> row gout0 + l
    int *status;
    int lat_t, abs_t;
    int B, T, Gtot, g0, Gs, H, r;
    int L_lat;                   // cached tokens per sequence
    int L_out;                   // positions per score row (scan: L_lat; gather: m)
    int n_gather;                // valid gathered positions (gather mode)
    int Gout = 0;                // score rows per (sequence, query); 0 = Gs
    int gout0 = 0;               // first of them written by this launch
};
cudaError_t launch_score_simt(const ScoreParams &p, cudaStream_t s);
bool score_tc_supported(const ScoreParams &p);
cudaError_t launch_score_tc(const ScoreParams &p, cudaStream_t s);

// ------------------------------------------------------------- selection
// Row r of the input is scores + r * in_stride, with valid length
// valid_len[r] (or L_row); its selection goes to out row
//   (r / rows_per_group) * group_stride + (r % rows_per_group) + row_offset
// of idx/vals (each out row holds k entries).  When `map` is set, selected
// positions j are written as map[(r / rows_per_group) * map_stride + j].
struct TopkParams {
    const float *scores;
    int64_t rows;
    int64_t in_stride;
    int L_row;
    const int32_t *valid_len;
    int k;
    int32_t *idx;
    float *vals;
    int rows_per_group, group_stride, row_offset;
    const int32_t *map;
    int64_t map_stride;
    int *status;
    // segmented rows (first pass of the two-pass long-row selection): row i is
    // positions [s * seg_len, (s + 1) * seg_len) of score row i / segs,
    // s = i % segs; outputs are positions in the whole row.  Needs map and
    // valid_len NULL.
    int segs = 1;
    int seg_len = 0;
    int pad_idx = -1;   // index written to output slots past min(k, V)
    int64_t vals_stride = 0;   // floats between out rows of vals (0: k)
};
cudaError_t launch_topk(const TopkParams &p, cudaStream_t s);
// True when launch_topk spreads each row over a thread-block cluster (few
// rows longer than 8,192 scores, no candidate list, no segments): the
// two-pass workspace path is then not needed.
bool topk_cluster_path(const TopkParams &p);
// Longest row (and segment) the register-resident top-k takes.
constexpr int kTopkRegRow = 32768;

// Launches `kern` on stream `s` with programmatic stream serialization: the
// kernel may be scheduled while its predecessor in the stream finishes.  The
// library's kernels execute griddepcontrol.wait (griddep_wait) before their
// first global memory access, so only their set-up (shared memory, barriers,
// tensor memory) overlaps the predecessor; a decode scan's producer also
// issues its first latent loads (see griddep_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Per-device status word (address of the __device__ variable on the current
// device), or nullptr on failure.
int *device_status_ptr();

// The argument checks of li_hs_select other than its workspace (LI_OK or the
// error status), shared with the entry points that supply their own scratch.
int hs_check_args(const void *latent, int lat_t, const float *lat_scale, const void *q_abs,
                  int abs_t, const float *q_abs_scale, const float *w, const float *beta, int B,
                  int G, int H, int r, int L, int m, int k, const int32_t *cand, const int32_t *idx);

} // namespace li
