// score_tc.cu -- group scoring on the tensor cores (tcgen05 + TMA + TMEM).
//
// Computes eq. (8) of "LatentIndex: Cross-Layer Sharing with Layer-Specific
// Selection for Sparse Attention" (summary page, Methodology):
//     u_l(t) = sum_h w_{l,h} ReLU(q~_{l,h} . c_t + beta_{l,h})
// for Gs layers at once.  The dot products of one sequence/query are the dense
// contraction  [128 cached tokens x r] x [r x N],  N = Gs*H absorbed heads,
// which is exactly one tcgen05.mma tile shape (M = 128, N <= 256): the tokens
// sit on M so that TMEM lane i holds token i with all its N head columns, and
// the ReLU / weighted head reduction of eq. (8) becomes a per-thread loop over
// TMEM columns in the epilogue (no shuffles), one coalesced score store per
// layer.
//
// Scaled fp8 storage: the latent row t and the absorbed row (l,h) carry fp32
// scales s_c(t), s_q(l,h) >= 0, so  q~.c = s_q s_c (code_q . code_c)  and,
// with beta = 0,  w ReLU(s_q s_c a) = s_c (w s_q) ReLU(a): the scales leave
// the inner loop (w s_q is precomputed per query, s_c applied once per token).
// With beta the scales are applied before the ReLU.
//
// Roles of the 384 threads (one persistent CTA per SM, static contiguous
// split of the (query, 128-token tile) work units):
//   warp 0      TMA producer: latent tiles -> smem ring (and the query
//               operand whenever the work unit's query changes)
//   warp 1      TMEM allocation and the single-thread MMA issuer
//   warps 2-3   gather mode only: with warp 0, copy gathered latent rows
//               into the swizzled smem layout (HS followers rescoring the
//               anchor's candidates)
//   warps 4-11  epilogue, two warps per TMEM lane quarter (warp % 4), each
//               taking half of the layers: TMEM -> registers 32 columns at a
//               time (the next chunk's load in flight while the current one
//               is reduced), ReLU, weighted head sums with packed fp32 FMA,
//               per-token scale, one coalesced score store per layer
// The two TMEM accumulators are double-buffered so the epilogue of tile i
// overlaps the MMAs of tile i+1 and the loads of the tiles after it.
//
// Operand layouts: K-major, split in 64-element K chunks; bf16 chunks are
// 128-byte rows (128B swizzle), fp8 chunks 64-byte rows (64B swizzle); an
// 8-row group spans 1024 / 512 bytes (the descriptors' stride byte offset).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "li_internal.cuh"
#include "ptx.cuh"

namespace li {
namespace {

constexpr int kThreads = 384;
constexpr int kEpiWarps = 8;
constexpr int kTileM = 128;
constexpr int kChunkElems = 64;
constexpr int kMaxDev = 64;
constexpr int kSmemBudget = 200 * 1024;

struct TcConfig {
    int N;              // Gs * H
    int nchunk;         // r / 64
    int stages;
    int a_chunk_bytes;  // 128 * 64 * esz
    int b_chunk_bytes;  // N * 64 * esz
    int a_stage_bytes;
    int off_a;          // byte offsets from the 1024-aligned base
    int off_bar;
    int off_misc;
    int tmem_cols;
    int acc_stride;     // TMEM column distance of the two accumulators
    int NT;             // tiles per query row
    int64_t U;          // total work units
};

struct __align__(8) Bars {
    uint64_t b_full, b_empty, done;
    uint64_t tmem_full[2], tmem_empty[2];
};

struct Misc {
    uint32_t tmem_base;
    int abort;
    int pad[2];
    // per-epilogue-warp copies of the current query's head constants for the
    // warp's layers (<= 128 columns), so no cross-warp barrier is needed when
    // the query changes
    float wq[kEpiWarps][128];
    float sq[kEpiWarps][128];
    float bq[kEpiWarps][128];
};

// One lane polls, the whole warp gets the (uniform) outcome.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          int *status)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0)
        ok = mbar_wait(bar, parity, abort, status, kWaitLimitNs);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Walks a CTA's contiguous range of (query row bt, 128-token tile) work units
// without a 64-bit division per unit.
struct UnitIter {
    int64_t bt;
    int tile;
    int NT;
    __device__ __forceinline__ UnitIter(int64_t u, int nt) : bt(u / nt), tile(static_cast<int>(u % nt)), NT(nt) {}
    __device__ __forceinline__ void next()
    {
        if (++tile == NT) {
            tile = 0;
            ++bt;
        }
    }
};

__device__ __forceinline__ int seq_of(int64_t bt, int T)
{
    return T == 1 ? static_cast<int>(bt) : static_cast<int>(bt / T);
}

template <bool kGather>
__device__ __forceinline__ int unit_valid_len(const ScoreParams &p, int64_t bt)
{
    if (kGather)
        return p.n_gather;
    if (p.q_pos == nullptr)
        return p.L_lat;
    int t = static_cast<int>(bt % p.T);
    int lim = p.q_pos[t] + 1;
    return lim < p.L_lat ? lim : p.L_lat;
}

template <bool kFP8, bool kGather, bool kBeta, int kH>
__global__ void __launch_bounds__(kThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const ScoreParams p, const TcConfig c)
{
    constexpr int kEsz = kFP8 ? 1 : 2;
    constexpr int kKStep = 32 / kEsz;              // elements per MMA K step (32 bytes)
    constexpr int kStepsPerChunk = kChunkElems / kKStep;
    constexpr uint32_t kSwz = kFP8 ? 4u : 2u;      // 64B : 128B swizzle
    constexpr uint32_t kSbo = 8u * kChunkElems * kEsz;
    constexpr int kPiece = 16;                     // bytes per gather copy
    constexpr int kPiecesPerChunk = kChunkElems * kEsz / kPiece;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *base = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
    uint8_t *smB = base;
    uint8_t *smA = base + c.off_a;
    uint64_t *full = reinterpret_cast<uint64_t *>(base + c.off_bar);
    uint64_t *empty = full + c.stages;
    Bars *bars = reinterpret_cast<Bars *>(empty + c.stages);
    Misc *misc = reinterpret_cast<Misc *>(base + c.off_misc);
    volatile int *abort_flag = &misc->abort;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int64_t u_begin = static_cast<int64_t>(blockIdx.x) * c.U / gridDim.x;
    const int64_t u_end = static_cast<int64_t>(blockIdx.x + 1) * c.U / gridDim.x;
    const int Gs = p.Gs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < c.stages; ++s) {
            mbar_init(&full[s], kGather ? 3u : 1u);
            mbar_init(&empty[s], 1u);
        }
        mbar_init(&bars->b_full, 1u);
        mbar_init(&bars->b_empty, 1u);
        mbar_init(&bars->done, 1u);
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bars->tmem_full[a], 1u);
            mbar_init(&bars->tmem_empty[a], static_cast<uint32_t>(kEpiWarps));
        }
        misc->abort = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(&misc->tmem_base, static_cast<uint32_t>(c.tmem_cols));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc->tmem_base;

    if (!kGather && warp == 0) {
        // ------------------------------------------------- TMA producer (1 thread)
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            int stage = 0;
            uint32_t phase = 0;
            int64_t cur_bt = -1;
            int nb = 0;
            uint32_t last_par[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            bool used[8] = {false, false, false, false, false, false, false, false};
            UnitIter it(u_begin, c.NT);
            for (int64_t u = u_begin; u < u_end; ++u, it.next()) {
                const int64_t bt = it.bt;
                const int tile = it.tile;
                if (tile * kTileM >= unit_valid_len<kGather>(p, bt))
                    continue;
                if (bt != cur_bt) {
                    if (nb > 0 && !mbar_wait(&bars->b_empty, (nb - 1) & 1, abort_flag, p.status,
                                             kWaitLimitNs))
                        break;
                    mbar_arrive_expect_tx(&bars->b_full,
                                          static_cast<uint32_t>(c.nchunk * c.b_chunk_bytes));
                    const int row0 = static_cast<int>((bt * p.Gtot + p.g0) * p.H);
                    for (int ch = 0; ch < c.nchunk; ++ch)
                        tma_load_2d(smB + ch * c.b_chunk_bytes, &tmB, &bars->b_full,
                                    ch * kChunkElems, row0);
                    cur_bt = bt;
                    ++nb;
                }
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, kWaitLimitNs))
                    break;
                uint8_t *dstA = smA + stage * c.a_stage_bytes;
                mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(c.a_stage_bytes));
                const int b = seq_of(bt, p.T);
                for (int ch = 0; ch < c.nchunk; ++ch)
                    tma_load_3d(dstA + ch * c.a_chunk_bytes, &tmA, &full[stage], ch * kChunkElems,
                                tile * kTileM, b);
                used[stage] = true;
                last_par[stage] = phase;
                if (++stage == c.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // Never leave the CTA with copies in flight: wait (bounded) for the
            // last load issued into each stage and for the last query operand.
            for (int s2 = 0; s2 < c.stages; ++s2)
                if (used[s2])
                    mbar_wait(&full[s2], last_par[s2], abort_flag, p.status, kWaitLimitNs);
            if (nb > 0)
                mbar_wait(&bars->b_full, (nb - 1) & 1, abort_flag, p.status, kWaitLimitNs);
        }
        __syncwarp();
    } else if (kGather && (warp == 0 || warp == 2 || warp == 3)) {
        // ------------------------------- gather producer (3 warps, 96 threads)
        // Copies the rows of the gathered token indices into the same swizzled
        // K-major layout TMA would write; warp 0 lane 0 also loads the query
        // operand by TMA.  All decisions are warp-uniform.
        const int pid = (warp == 0 ? 0 : warp - 1) * 32 + lane;
        if (warp == 0 && lane == 0)
            tma_prefetch_desc(&tmB);
        int stage = 0;
        uint32_t phase = 0;
        int64_t cur_bt = -1;
        int nb = 0;
        const int pieces_per_row = c.nchunk * kPiecesPerChunk;
        const int total = kTileM * pieces_per_row;
        const uint8_t *lat = static_cast<const uint8_t *>(p.latent);
        UnitIter it(u_begin, c.NT);
        for (int64_t u = u_begin; u < u_end; ++u, it.next()) {
            const int64_t bt = it.bt;
            const int tile = it.tile;
            if (tile * kTileM >= unit_valid_len<kGather>(p, bt))
                continue;
            const int b = seq_of(bt, p.T);
            if (bt != cur_bt) {
                if (warp == 0) {
                    bool ok = true;
                    if (lane == 0) {
                        if (nb > 0)
                            ok = mbar_wait(&bars->b_empty, (nb - 1) & 1, abort_flag, p.status,
                                           kWaitLimitNs);
                        if (ok) {
                            mbar_arrive_expect_tx(&bars->b_full,
                                                  static_cast<uint32_t>(c.nchunk * c.b_chunk_bytes));
                            const int row0 = static_cast<int>((bt * p.Gtot + p.g0) * p.H);
                            for (int ch = 0; ch < c.nchunk; ++ch)
                                tma_load_2d(smB + ch * c.b_chunk_bytes, &tmB, &bars->b_full,
                                            ch * kChunkElems, row0);
                        }
                    }
                    if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0)
                        break;
                }
                cur_bt = bt;
                ++nb;
            }
            if (!warp_wait(&empty[stage], phase ^ 1u, abort_flag, p.status))
                break;
            uint8_t *dstA = smA + stage * c.a_stage_bytes;
            const int32_t *gidx = p.gather_idx + static_cast<int64_t>(b) * p.L_out;
            for (int q = pid; q < total; q += 96) {
                const int row = q / pieces_per_row;
                const int j = q % pieces_per_row;
                const int ch = j / kPiecesPerChunk;
                const int qc = j % kPiecesPerChunk;
                const int slot = tile * kTileM + row;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (slot < p.n_gather) {
                    const int idx = __ldg(gidx + slot);
                    if (idx >= 0 && idx < p.L_lat) {
                        const uint8_t *src = lat +
                                             ((static_cast<int64_t>(b) * p.L_lat + idx) * p.r +
                                              ch * kChunkElems) * kEsz + qc * kPiece;
                        v = __ldg(reinterpret_cast<const uint4 *>(src));
                    } else {
                        atomicCAS(p.status, 0, -7 /* LI_ERR_DEVICE_BOUNDS */);
                    }
                }
                uint32_t off = static_cast<uint32_t>(row * (kChunkElems * kEsz) + qc * kPiece);
                off ^= ((off >> 7) & (kFP8 ? 3u : 7u)) << 4;
                *reinterpret_cast<uint4 *>(dstA + ch * c.a_chunk_bytes + off) = v;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&full[stage]);
            if (++stage == c.stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (warp == 0 && lane == 0 && nb > 0)
            mbar_wait(&bars->b_full, (nb - 1) & 1, abort_flag, p.status, kWaitLimitNs);
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = umma_idesc(kFP8, kTileM, c.N);
            const uint32_t a_base = smem_u32(smA);
            const uint32_t b_base = smem_u32(smB);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int64_t cur_bt = -1;
            int nb = 0;
            UnitIter it(u_begin, c.NT);
            for (int64_t u = u_begin; u < u_end; ++u, it.next()) {
                const int64_t bt = it.bt;
                const int tile = it.tile;
                if (tile * kTileM >= unit_valid_len<kGather>(p, bt))
                    continue;
                if (bt != cur_bt) {
                    if (nb > 0)
                        umma_commit(&bars->b_empty);
                    if (!mbar_wait(&bars->b_full, nb & 1, abort_flag, p.status, kWaitLimitNs))
                        break;
                    cur_bt = bt;
                    ++nb;
                }
                if (!mbar_wait(&bars->tmem_empty[acc], acc_phase ^ 1u, abort_flag, p.status,
                               kWaitLimitNs))
                    break;
                if (!mbar_wait(&full[stage], phase, abort_flag, p.status, kWaitLimitNs))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * c.acc_stride);
                const uint32_t a_stage = a_base + static_cast<uint32_t>(stage * c.a_stage_bytes);
                for (int ch = 0; ch < c.nchunk; ++ch) {
#pragma unroll
                    for (int ks = 0; ks < kStepsPerChunk; ++ks) {
                        const uint64_t ad = umma_sdesc(
                            a_stage + static_cast<uint32_t>(ch * c.a_chunk_bytes + ks * 32), kSbo, kSwz);
                        const uint64_t bd = umma_sdesc(
                            b_base + static_cast<uint32_t>(ch * c.b_chunk_bytes + ks * 32), kSbo, kSwz);
                        const uint32_t accum = (ch | ks) != 0 ? 1u : 0u;
                        if (kFP8)
                            umma_fp8(d_tmem, ad, bd, idesc, accum);
                        else
                            umma_bf16(d_tmem, ad, bd, idesc, accum);
                    }
                }
                umma_commit(&empty[stage]);
                umma_commit(&bars->tmem_full[acc]);
                if (++stage == c.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
                acc ^= 1;
                if (acc == 0)
                    acc_phase ^= 1u;
            }
            // all MMAs issued by this thread have completed before TMEM is freed
            umma_commit(&bars->done);
            mbar_wait(&bars->done, 0, abort_flag, p.status, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        constexpr int CH = kH < 32 ? kH : 32;          // TMEM columns per load
        constexpr int CPL = kH / CH;                   // loads per layer
        const int e = warp - 4;                        // 0..7
        const int quarter = warp & 3;                  // TMEM lane quarter
        const int lper = (Gs + 1) / 2;
        const int l_begin = (e >> 2) * lper;
        const int l_end = min(Gs, l_begin + lper);
        const int nlay = l_end > l_begin ? l_end - l_begin : 0;
        const int nchunks = nlay * CPL;
        const int row = quarter * 32 + lane;
        float *wq = misc->wq[e];
        float *sq = misc->sq[e];
        float *bq = misc->bq[e];
        int acc = 0;
        uint32_t acc_phase = 0;
        int64_t cur_bt = -1;
        UnitIter it(u_begin, c.NT);
        for (int64_t u = u_begin; u < u_end; ++u, it.next()) {
            const int64_t bt = it.bt;
            const int tile = it.tile;
            const int Lv = unit_valid_len<kGather>(p, bt);
            if (tile * kTileM >= Lv)
                continue;
            const int b = seq_of(bt, p.T);
            if (bt != cur_bt) {
                __syncwarp();
                const int64_t wrow = (bt * p.Gtot + p.g0 + l_begin) * p.H;
                for (int j = lane; j < nlay * kH; j += 32) {
                    const float wv = p.w[wrow + j];
                    const float sv = p.q_abs_scale ? p.q_abs_scale[wrow + j] : 1.f;
                    if (kBeta) {
                        wq[j] = wv;
                        sq[j] = sv;
                        bq[j] = p.beta[wrow + j];
                    } else {
                        wq[j] = wv * sv;
                    }
                }
                __syncwarp();
                cur_bt = bt;
            }
            if (!warp_wait(&bars->tmem_full[acc], acc_phase, abort_flag, p.status))
                break;
            tc_fence_after();
            const int pos = tile * kTileM + row;
            const bool valid = pos < Lv;
            float sc = 1.f;
            if (p.lat_scale != nullptr) {
                sc = 0.f;
                if (valid) {
                    int tok = pos;
                    if (kGather)
                        tok = p.gather_idx[static_cast<int64_t>(b) * p.L_out + pos];
                    if (tok >= 0 && tok < p.L_lat)
                        sc = p.lat_scale[static_cast<int64_t>(b) * p.L_lat + tok];
                }
            }
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc * c.acc_stride + l_begin * kH);
            float *out = p.scores + (bt * Gs + l_begin) * static_cast<int64_t>(p.L_out) + pos;

            float2 s2a = make_float2(0.f, 0.f), s2b = make_float2(0.f, 0.f);
            // reduce one chunk of CH head columns into the running layer sum
            auto consume = [&](int i, const uint32_t (&v)[CH]) {
                const int col = i * CH;
                if (kBeta) {
#pragma unroll
                    for (int j = 0; j < CH; j += 2) {
                        const float x0 = fmaf(__uint_as_float(v[j]) * sq[col + j], sc, bq[col + j]);
                        const float x1 = fmaf(__uint_as_float(v[j + 1]) * sq[col + j + 1], sc, bq[col + j + 1]);
                        s2a = __ffma2_rn(make_float2(wq[col + j], wq[col + j + 1]),
                                         make_float2(fmaxf(x0, 0.f), fmaxf(x1, 0.f)), s2a);
                    }
                } else {
                    const float4 *w4 = reinterpret_cast<const float4 *>(wq + col);
#pragma unroll
                    for (int j = 0; j < CH; j += 4) {
                        const float4 ww = w4[j / 4];
                        s2a = __ffma2_rn(make_float2(ww.x, ww.y),
                                         make_float2(fmaxf(__uint_as_float(v[j]), 0.f),
                                                     fmaxf(__uint_as_float(v[j + 1]), 0.f)), s2a);
                        s2b = __ffma2_rn(make_float2(ww.z, ww.w),
                                         make_float2(fmaxf(__uint_as_float(v[j + 2]), 0.f),
                                                     fmaxf(__uint_as_float(v[j + 3]), 0.f)), s2b);
                    }
                }
                if ((i + 1) % CPL == 0) {
                    float uval = (s2a.x + s2a.y) + (s2b.x + s2b.y);
                    if (!kBeta)
                        uval *= sc;
                    if (valid)
                        out[static_cast<int64_t>(i / CPL) * p.L_out] = uval;
                    s2a = make_float2(0.f, 0.f);
                    s2b = make_float2(0.f, 0.f);
                }
            };
            uint32_t va[CH], vb[CH];
            if (nchunks > 0)
                tmem_ld_chunk(tbase, va);
            for (int i = 0; i < nchunks; i += 2) {
                tmem_wait_chunk(va);
                if (i + 1 < nchunks)
                    tmem_ld_chunk(tbase + static_cast<uint32_t>((i + 1) * CH), vb);
                consume(i, va);
                if (i + 1 < nchunks) {
                    tmem_wait_chunk(vb);
                    if (i + 2 < nchunks)
                        tmem_ld_chunk(tbase + static_cast<uint32_t>((i + 2) * CH), va);
                    consume(i + 1, vb);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->tmem_empty[acc]);
            acc ^= 1;
            if (acc == 0)
                acc_phase ^= 1u;
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, static_cast<uint32_t>(c.tmem_cols));
    }
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

int sm_count()
{
    static std::atomic<int> cache[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return 148;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

bool make_config(const ScoreParams &p, bool fp8, TcConfig &c, int &smem_bytes)
{
    const int esz = fp8 ? 1 : 2;
    c.N = p.Gs * p.H;
    c.nchunk = p.r / kChunkElems;
    c.a_chunk_bytes = kTileM * kChunkElems * esz;
    c.b_chunk_bytes = c.N * kChunkElems * esz;
    c.a_stage_bytes = c.nchunk * c.a_chunk_bytes;
    const int b_bytes = c.nchunk * c.b_chunk_bytes;
    const int b_bytes_al = (b_bytes + 1023) & ~1023;
    int stages = (kSmemBudget - b_bytes_al - 4096) / c.a_stage_bytes;
    if (stages > 8)
        stages = 8;
    if (stages < 2)
        return false;
    c.stages = stages;
    c.off_a = b_bytes_al;
    c.off_bar = c.off_a + stages * c.a_stage_bytes;
    const int bar_bytes = 2 * stages * 8 + static_cast<int>(sizeof(Bars));
    c.off_misc = (c.off_bar + bar_bytes + 15) & ~15;
    smem_bytes = c.off_misc + static_cast<int>(sizeof(Misc)) + 1024;
    // one CTA per SM: a second CTA would only queue on the TMEM allocation
    if (smem_bytes < 116 * 1024)
        smem_bytes = 116 * 1024;
    int cols = 32;
    while (cols < 2 * c.N)
        cols <<= 1;
    c.tmem_cols = cols;
    c.acc_stride = cols / 2;
    const int Lrow = p.gather_idx ? p.L_out : p.L_lat;
    c.NT = (Lrow + kTileM - 1) / kTileM;
    c.U = static_cast<int64_t>(p.B) * p.T * c.NT;
    return smem_bytes <= 227 * 1024 && cols <= 512;
}

template <bool kFP8, bool kGather, bool kBeta, int kH>
cudaError_t launch_t(const CUtensorMap &tmA, const CUtensorMap &tmB, const ScoreParams &p,
                     const TcConfig &c, int smem_bytes, cudaStream_t s)
{
    auto kern = score_tc_kernel<kFP8, kGather, kBeta, kH>;
    static std::atomic<int> set_bytes[kMaxDev];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDev)
        dev = 0;
    if (set_bytes[dev].load(std::memory_order_relaxed) < smem_bytes) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e != cudaSuccess)
            return e;
        set_bytes[dev].store(227 * 1024, std::memory_order_relaxed);
    }
    int64_t grid = sm_count();
    if (grid > c.U)
        grid = c.U;
    if (grid <= 0)
        return cudaSuccess;
    kern<<<static_cast<unsigned>(grid), kThreads, smem_bytes, s>>>(tmA, tmB, p, c);
    return cudaGetLastError();
}

template <bool kFP8, bool kGather, bool kBeta>
cudaError_t dispatch_h(const CUtensorMap &tmA, const CUtensorMap &tmB, const ScoreParams &p,
                       const TcConfig &c, int smem_bytes, cudaStream_t s)
{
    switch (p.H) {
    case 16: return launch_t<kFP8, kGather, kBeta, 16>(tmA, tmB, p, c, smem_bytes, s);
    case 32: return launch_t<kFP8, kGather, kBeta, 32>(tmA, tmB, p, c, smem_bytes, s);
    case 64: return launch_t<kFP8, kGather, kBeta, 64>(tmA, tmB, p, c, smem_bytes, s);
    case 128: return launch_t<kFP8, kGather, kBeta, 128>(tmA, tmB, p, c, smem_bytes, s);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace

bool score_tc_supported(const ScoreParams &p)
{
    const bool fp8 = p.lat_t == LI_FP8_E4M3 && p.abs_t == LI_FP8_E4M3;
    const bool bf16 = p.lat_t == LI_BF16 && p.abs_t == LI_BF16;
    if (!fp8 && !bf16)
        return false;
    if (p.r % kChunkElems != 0 || p.r > 256)
        return false;
    if (p.H != 16 && p.H != 32 && p.H != 64 && p.H != 128)
        return false;
    const int N = p.Gs * p.H;
    if (N < 16 || N > 256 || N % 16 != 0)
        return false;
    if (p.gather_idx != nullptr && p.q_pos != nullptr)
        return false;
    if (static_cast<int64_t>(p.B) * p.T * p.Gtot * p.H > 0x7FFFFFFF || p.L_lat > 0x7FFFFFFF / 2)
        return false;
    TcConfig c;
    int smem = 0;
    return make_config(p, fp8, c, smem) && encode_fn() != nullptr;
}

cudaError_t launch_score_tc(const ScoreParams &p, cudaStream_t s)
{
    const bool fp8 = p.lat_t == LI_FP8_E4M3;
    const bool gather = p.gather_idx != nullptr;
    TcConfig c;
    int smem_bytes = 0;
    if (!make_config(p, fp8, c, smem_bytes))
        return cudaErrorInvalidValue;
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr)
        return cudaErrorNotSupported;
    const int esz = fp8 ? 1 : 2;
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapSwizzle swz = fp8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;

    CUtensorMap tmA, tmB;
    // latent [B][L][r] as a 3D map {r, L, B}; box {64, 128, 1}
    {
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(p.r), static_cast<cuuint64_t>(p.L_lat),
                              static_cast<cuuint64_t>(p.B)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(p.r) * esz,
                                 static_cast<cuuint64_t>(p.r) * esz * p.L_lat};
        cuuint32_t box[3] = {kChunkElems, kTileM, 1};
        cuuint32_t estr[3] = {1, 1, 1};
        if (enc(&tmA, dt, 3, const_cast<void *>(p.latent), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // absorbed queries [B*T*Gtot*H][r] as a 2D map; box {64, N}
    {
        cuuint64_t rows = static_cast<cuuint64_t>(p.B) * p.T * p.Gtot * p.H;
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.r), rows};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.r) * esz};
        cuuint32_t box[2] = {kChunkElems, static_cast<cuuint32_t>(c.N)};
        cuuint32_t estr[2] = {1, 1};
        if (enc(&tmB, dt, 2, const_cast<void *>(p.q_abs), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const bool beta = p.beta != nullptr;
    if (fp8) {
        if (gather)
            return beta ? dispatch_h<true, true, true>(tmA, tmB, p, c, smem_bytes, s)
                        : dispatch_h<true, true, false>(tmA, tmB, p, c, smem_bytes, s);
        return beta ? dispatch_h<true, false, true>(tmA, tmB, p, c, smem_bytes, s)
                    : dispatch_h<true, false, false>(tmA, tmB, p, c, smem_bytes, s);
    }
    if (gather)
        return beta ? dispatch_h<false, true, true>(tmA, tmB, p, c, smem_bytes, s)
                    : dispatch_h<false, true, false>(tmA, tmB, p, c, smem_bytes, s);
    return beta ? dispatch_h<false, false, true>(tmA, tmB, p, c, smem_bytes, s)
                : dispatch_h<false, false, false>(tmA, tmB, p, c, smem_bytes, s);
}

} // namespace li
