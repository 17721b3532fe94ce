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
// Roles (one persistent CTA per SM, static contiguous split of the
// (query row, 128-token tile) work units; every role walks the same units):
//   warp 0          TMEM allocation; MMA issuer of the CTA's even tiles
//   warp after the producers: MMA issuer of the odd tiles (two issuers keep
//                   one tile's MMAs queued while the other's execute)
//   warp 1          scan mode: TMA producer of the latent tiles (smem ring),
//                   of each tile's 128 fp32 token scales (fp8 latents; into
//                   the same stage, on the same barrier) and of the absorbed-query
//                   operand (double-buffered when it fits, so the next
//                   query's operand loads under the current query's tiles)
//   warps 1-2       gather mode (HS followers rescoring the anchor's
//                   candidates): each thread copies two tile rows of gathered
//                   latent with 16-byte cp.async into the swizzled layout TMA
//                   would write, several tiles in flight per thread
//   16 warps        epilogue (8 at H = 128), four per TMEM lane quarter
//                   (warp % 4), each owning 64 accumulator columns (one layer
//                   at H = 64; 128 columns at H = 128): its columns in flight
//                   at once, the accumulator released as soon as they land,
//                   then ReLU, weighted head sums with packed fp32 FMA, the
//                   token's scale (read from the stage, which is then handed
//                   back) and one coalesced store per layer.
// The epilogue sets the tile period: each warp's chain per tile is wait,
// accumulator load, arithmetic, store.  Measured with per-role clock stamps
// (32 sequences x 32K, fp8): the MMAs of the next tile are complete before
// the epilogue has released the current one.  Two changes shortened that
// chain: the token scales arrive with the tile (a global load issued one tile
// ahead cost a full HBM round trip per tile), and 64 instead of 128 columns
// per warp halve its arithmetic.
// The two TMEM accumulators (2 x 256 columns) are double-buffered so the
// epilogue of tile i overlaps the MMAs of tile i+1 and the loads of the tiles
// after it.
//
// Operand layouts: K-major, split in 64-element K chunks; bf16 chunks are
// 128-byte rows (128B swizzle), fp8 chunks 64-byte rows (64B swizzle); an
// 8-row group spans 1024 / 512 bytes (the descriptors' stride byte offset).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "li_internal.cuh"
#include "ptx.cuh"

namespace li {
namespace {

constexpr int kTileM = 128;
constexpr int kChunkElems = 64;
constexpr int kMaxDev = 64;
constexpr int kTmemCols = 512;          // two accumulators of 256 columns
constexpr int kAccStride = 256;
constexpr int kConstCap = 1024;         // active epilogue warps x columns per warp
constexpr int kScRing = 4;              // token-scale slots handed from the MMA warps to the epilogue
constexpr int kSmemLimit = 227 * 1024;

// Epilogue warps own 64 accumulator columns each (one layer at H = 64), four
// per 64-column block (one per TMEM lane quarter); at H = 128 a layer's
// weighted sum spans 128 columns, so its warps own 128.
template <int kH>
struct EpiShape {
    static constexpr int kCols = kH == 128 ? 128 : 64;
    static constexpr int kWarps = 4 * (256 / kCols);
};

template <bool kGather, int kH>
struct Roles {
    static constexpr int kMmaWarp = 0;                        // even tiles (accumulator 0)
    static constexpr int kProdWarp0 = 1;
    static constexpr int kProdWarps = kGather ? 2 : 1;
    static constexpr int kMmaWarp1 = kProdWarp0 + kProdWarps;  // odd tiles (accumulator 1)
    static constexpr int kEpiWarp0 = kMmaWarp1 + 1;
    static constexpr int kEpiWarps = EpiShape<kH>::kWarps;
    static constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
};

struct TcConfig {
    int N;              // Gs * H
    int nchunk;         // r / 64
    int stages;         // latent tile ring depth
    int nbuf;           // query-operand buffers (1 or 2)
    int a_chunk_bytes;  // 128 * 64 * esz
    int b_chunk_bytes;  // N * 64 * esz
    int a_stage_bytes;
    int b_bytes;        // one query operand
    int b_buf_stride;   // 1024-aligned
    int off_a;          // byte offsets from the 1024-aligned base
    int off_sc;         // per-stage token scales (sc_stage)
    int off_bar;
    int off_misc;
    int cw;             // accumulator columns per epilogue warp
    int nepi;           // epilogue warps with columns
    int sc_stage;       // the latent's per-token scales travel with each tile (TMA into the stage)
    int sc_ring;        // ... and leave the stage with the tile's MMA warp for a ring slot
                        // (shallow latent rings), else the epilogue reads them in the stage
    int gdepth;         // gather mode: tiles in flight per copying thread
    int NT;             // tiles per query row
    int64_t U;          // total work units
};

struct __align__(8) Bars {
    uint64_t b_full[2], b_empty[2];
    uint64_t tmem_full[2], tmem_empty[2];
    uint64_t done;
};

struct Misc {
    uint32_t tmem_base;
    int abort;
    int pad[2];
    // per-epilogue-warp copies of the current query's head constants for the
    // warp's columns, so that no cross-warp barrier is needed when the query
    // changes
    float wq[kConstCap];
    float sq[kConstCap];
    float bq[kConstCap];
    // token scales of the CTA's tiles ord % kScRing, copied out of the latent
    // stage by the tile's MMA warp (sc_stage)
    __align__(16) float scr[kScRing][kTileM];
};

// The whole (converged) warp waits; the outcome is made warp-uniform, so that
// a warp never splits on a wait that ran out.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          int *status)
{
    bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok))
        return true;
    ok = ok || mbar_wait(bar, parity, abort, status, kWaitLimitNs);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ int seq_of(int bt, int T)
{
    return T == 1 ? bt : bt / T;
}

template <bool kGather>
__device__ __forceinline__ int unit_valid_len(const ScoreParams &p, int bt)
{
    if (kGather)
        return p.n_gather;
    if (p.q_pos == nullptr)
        return p.L_lat;
    const int t = bt % p.T;
    const int lim = p.q_pos[t] + 1;
    return lim < p.L_lat ? lim : p.L_lat;
}

// Walks a CTA's contiguous range of (query row bt, 128-token tile) work units,
// skipping tiles that lie entirely past the row's valid length (causal
// prefill), without a division per unit.  `left` counts the units of the
// range from the current one on.
template <bool kGather>
struct Walk {
    int left, bt, tile, Lv;

    __device__ __forceinline__ void init(const ScoreParams &p, int64_t ub, int64_t ue, int NT)
    {
        left = static_cast<int>(ue - ub);
        bt = static_cast<int>(ub / NT);
        tile = static_cast<int>(ub % NT);
        Lv = left > 0 ? unit_valid_len<kGather>(p, bt) : 0;
        settle(p, NT);
    }
    __device__ __forceinline__ void settle(const ScoreParams &p, int NT)
    {
        while (left > 0 && tile * kTileM >= Lv) {
            left -= NT - tile;
            ++bt;
            tile = 0;
            if (left > 0)
                Lv = unit_valid_len<kGather>(p, bt);
        }
    }
    __device__ __forceinline__ bool ok() const { return left > 0; }
    __device__ __forceinline__ void next(const ScoreParams &p, int NT)
    {
        --left;
        if (++tile == NT) {
            tile = 0;
            ++bt;
            if (left > 0)
                Lv = unit_valid_len<kGather>(p, bt);
        }
        settle(p, NT);
    }
};

// Ties the registers of a finished tcgen05.ld to the preceding wait::ld (which
// covers every outstanding load of the thread) without another wait.
__device__ __forceinline__ void tmem_regs_ready(uint32_t (&v)[32])
{
    asm volatile(""
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_depth(int depth)
{
    if (depth <= 1)
        cp_async_wait_group<1>();
    else if (depth == 2)
        cp_async_wait_group<2>();
    else
        cp_async_wait_group<3>();
}

template <bool kFP8, bool kGather, bool kBeta, int kH>
__global__ void __launch_bounds__(Roles<kGather, kH>::kThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmS, const ScoreParams p, const TcConfig c)
{
    using R = Roles<kGather, kH>;
    constexpr int kEsz = kFP8 ? 1 : 2;
    constexpr int kKStep = 32 / kEsz;              // elements per MMA K step (32 bytes)
    constexpr int kStepsPerChunk = kChunkElems / kKStep;
    constexpr uint32_t kSwz = kFP8 ? 4u : 2u;      // 64B : 128B swizzle
    constexpr uint32_t kSbo = 8u * kChunkElems * kEsz;
    constexpr int kRowChunkBytes = kChunkElems * kEsz;
    constexpr int kPiecesPerChunk = kRowChunkBytes / 16;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *base = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
    uint8_t *smB = base;
    uint8_t *smA = base + c.off_a;
    float *smS = reinterpret_cast<float *>(base + c.off_sc);   // [stages][128] token scales
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
            mbar_init(&full[s], kGather ? static_cast<uint32_t>(R::kProdWarps) : 1u);
            // the MMAs' commit, and (scales read in the stage) each epilogue
            // warp once it has read the stage's token scales
            mbar_init(&empty[s], 1u + static_cast<uint32_t>(c.sc_stage && !c.sc_ring ? c.nepi : 0));
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bars->b_full[a], 1u);
            mbar_init(&bars->b_empty[a], 2u);      // one commit from each MMA warp
            // the MMAs' commit and, with the scale ring, the MMA warp once the
            // tile's scales are in their slot
            mbar_init(&bars->tmem_full[a], 1u + static_cast<uint32_t>(c.sc_ring));
            mbar_init(&bars->tmem_empty[a], static_cast<uint32_t>(c.nepi));
        }
        mbar_init(&bars->done, 2u);
        misc->abort = 0;
        mbar_fence_init();
    }
    if (warp == R::kMmaWarp) {
        tmem_alloc(&misc->tmem_base, static_cast<uint32_t>(kTmemCols));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc->tmem_base;
    // Each role waits for the preceding kernel (griddep_wait) before its first
    // global memory access, except the TMA producer of a decode scan, which
    // first issues the latent loads of its ring's first tiles: the latent cache
    // is not written by a kernel of this library that lets this one start early
    // (the append triggers its dependents only after its stores and a fence).
    griddep_launch_dependents();

    // Issues the query operand of row bt into buffer (nb % nbuf); returns false
    // on abort.  Called by a whole warp; lane 0 issues the copies.
    auto load_query_operand = [&](int bt, int nb) -> bool {
        const int bb = nb % c.nbuf;
        const int use = nb / c.nbuf;
        if (use > 0 &&
            !warp_wait(&bars->b_empty[bb], static_cast<uint32_t>(use - 1) & 1u, abort_flag, p.status))
            return false;
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars->b_full[bb], static_cast<uint32_t>(c.b_bytes));
            const int row0 = (bt * p.Gtot + p.g0) * p.H;
            uint8_t *dst = smB + bb * c.b_buf_stride;
            for (int ch = 0; ch < c.nchunk; ++ch)
                tma_load_2d(dst + ch * c.b_chunk_bytes, &tmB, &bars->b_full[bb], ch * kChunkElems, row0);
        }
        __syncwarp();
        return true;
    };
    // Never leave the CTA with query-operand copies in flight.
    auto drain_query_operand = [&](int nb) {
        for (int j = nb - 1; j >= 0 && j >= nb - c.nbuf; --j)
            mbar_wait(&bars->b_full[j % c.nbuf], static_cast<uint32_t>(j / c.nbuf) & 1u, abort_flag,
                      p.status, kWaitLimitNs);
    };

    if (warp == R::kMmaWarp || warp == R::kMmaWarp1) {
        // --------------------------------------------------------- MMA issuers
        // Two warps (on different SM sub-partitions) issue the MMAs: the first
        // the CTA's even tiles into accumulator 0, the second its odd tiles
        // into accumulator 1.  A tcgen05.mma issue stalls its warp until the
        // tensor pipe has room, which with one issuer meant that the next
        // tile's MMAs could not even be prepared while the current ones ran;
        // with two, one warp's MMAs are queued while the other's execute.
        // Both warps walk every unit (stage ring, query operand buffers), and
        // lane 0 issues the MMAs and commits.
        griddep_wait();
        const int par = warp == R::kMmaWarp ? 0 : 1;
        const uint32_t idesc = umma_idesc(kFP8, kTileM, c.N);
        const uint32_t a_base = smem_u32(smA);
        const uint32_t b_base0 = smem_u32(smB);
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(par * kAccStride);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t acc_phase = 0;
        int cur_bt = -1;
        int nb = 0;
        int ord = 0;                                   // tile ordinal within the CTA
        uint32_t b_base = b_base0;
        Walk<kGather> w;
        for (w.init(p, u_begin, u_end, c.NT); w.ok(); w.next(p, c.NT), ++ord) {
            if (w.bt != cur_bt) {
                if (nb > 0 && lane == 0)
                    umma_commit(&bars->b_empty[(nb - 1) % c.nbuf]);
                const int bb = nb % c.nbuf;
                if (!warp_wait(&bars->b_full[bb], static_cast<uint32_t>(nb / c.nbuf) & 1u, abort_flag,
                               p.status))
                    break;
                b_base = b_base0 + static_cast<uint32_t>(bb * c.b_buf_stride);
                cur_bt = w.bt;
                ++nb;
            }
            if ((ord & 1) == par) {
                if (!warp_wait(&bars->tmem_empty[par], acc_phase ^ 1u, abort_flag, p.status))
                    break;
                if (!warp_wait(&full[stage], phase, abort_flag, p.status))
                    break;
                tc_fence_after();
                if (c.sc_ring) {
                    // The tile's 128 token scales move to its ring slot, so that
                    // the stage is free again as soon as the MMAs have read it.
                    // Slot ord % kScRing was last read by the epilogue for tile
                    // ord - kScRing, which every epilogue warp did before it
                    // released tile ord - 2's accumulator (waited for above).
                    // The copy is published by an arrival on the accumulator's
                    // full barrier, whose phase then also waits for the MMAs'
                    // commit: one wait in the epilogue covers both.
                    const int sl = ord & (kScRing - 1);
                    reinterpret_cast<float4 *>(misc->scr[sl])[lane] =
                        reinterpret_cast<const float4 *>(smS + stage * kTileM)[lane];
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&bars->tmem_full[par]);
                }
                if (lane == 0) {
                    // descriptors of the stage's and the operand's first K step;
                    // later steps add their byte offset / 16 to the start-address
                    // field (shared addresses stay below 2^18, so it cannot carry)
                    const uint32_t a_stage = a_base + static_cast<uint32_t>(stage * c.a_stage_bytes);
                    const uint64_t ad0 = umma_sdesc(a_stage, kSbo, kSwz);
                    const uint64_t bd0 = umma_sdesc(b_base, kSbo, kSwz);
                    for (int ch = 0; ch < c.nchunk; ++ch) {
                        const uint64_t adc = ad0 + static_cast<uint64_t>((ch * c.a_chunk_bytes) >> 4);
                        const uint64_t bdc = bd0 + static_cast<uint64_t>((ch * c.b_chunk_bytes) >> 4);
#pragma unroll
                        for (int ks = 0; ks < kStepsPerChunk; ++ks) {
                            const uint64_t ad = adc + static_cast<uint64_t>(ks * 2);   // 32 bytes
                            const uint64_t bd = bdc + static_cast<uint64_t>(ks * 2);
                            const uint32_t accum = (ch | ks) != 0 ? 1u : 0u;
                            if (kFP8)
                                umma_fp8(d_tmem, ad, bd, idesc, accum);
                            else
                                umma_bf16(d_tmem, ad, bd, idesc, accum);
                        }
                    }
                    umma_commit(&empty[stage]);
                    umma_commit(&bars->tmem_full[par]);
                }
                __syncwarp();
                acc_phase ^= 1u;
            }
            if (++stage == c.stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        // all MMAs issued by lane 0 have completed before TMEM is freed
        if (lane == 0)
            umma_commit(&bars->done);
        __syncwarp();
        mbar_wait(&bars->done, 0, abort_flag, p.status, kWaitLimitNs);
        __syncwarp();
    } else if (!kGather && warp == R::kProdWarp0) {
        // ------------------------------------------------------ TMA producer
        // The warp walks the units together; lane 0 issues the copies.
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            if (c.sc_stage)
                tma_prefetch_desc(&tmS);
        }
        const uint64_t pol = make_l2_policy(p.T == 1);   // decode: each tile is read once
        int stage = 0;
        uint32_t phase = 0;
        int cur_bt = -1;
        int nb = 0;
        int issued = 0;
        // the latent (and scales) of tile `x` into its stage
        auto load_tile = [&](const Walk<kGather> &x, int st) {
            if (lane == 0) {
                uint8_t *dstA = smA + st * c.a_stage_bytes;
                mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(c.a_stage_bytes) +
                                                     (c.sc_stage ? kTileM * 4u : 0u));
                const int b = seq_of(x.bt, p.T);
                // all K chunks of the tile in one copy (the map's third
                // dimension is the chunk): [chunk][128 rows][64 elements]
                tma_load_4d_hint(dstA, &tmA, &full[st], 0, x.tile * kTileM, 0, b, pol);
                // the tile's 128 token scales (zero past the cache end)
                if (c.sc_stage)
                    tma_load_2d(smS + st * kTileM, &tmS, &full[st], x.tile * kTileM, b);
            }
            __syncwarp();
        };
        Walk<kGather> w;
        w.init(p, u_begin, u_end, c.NT);
        // Decode scans (no per-query causal limits to read): the ring's first
        // tiles before waiting for the preceding kernel; their stages are
        // still free.
        int pre = 0;
        if (p.q_pos == nullptr) {
            Walk<kGather> x = w;
            for (; x.ok() && pre < c.stages; x.next(p, c.NT), ++pre)
                load_tile(x, pre);
        }
        griddep_wait();
        for (; w.ok(); w.next(p, c.NT)) {
            if (w.bt != cur_bt) {
                if (!load_query_operand(w.bt, nb))
                    break;
                cur_bt = w.bt;
                ++nb;
            }
            if (issued >= pre) {                 // (the first `pre` were issued before the wait)
                if (!warp_wait(&empty[stage], phase ^ 1u, abort_flag, p.status))
                    break;
                load_tile(w, stage);
            }
            ++issued;
            if (++stage == c.stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        // Never leave the CTA with copies in flight: wait (bounded) for the
        // last load issued into each stage and for the last query operands
        // (the tiles issued before the wait count even when the loop stopped
        // before reaching them).
        if (issued < pre)
            issued = pre;
        for (int s2 = 0; s2 < c.stages && s2 < issued; ++s2) {
            const int last = s2 + (issued - 1 - s2) / c.stages * c.stages;   // last tile into s2
            mbar_wait(&full[s2], static_cast<uint32_t>(last / c.stages) & 1u, abort_flag, p.status,
                      kWaitLimitNs);
        }
        drain_query_operand(nb);
        __syncwarp();
    } else if (kGather && warp >= R::kProdWarp0 && warp < R::kProdWarp0 + R::kProdWarps) {
        griddep_wait();
        // ------------------------------- gather producer (2 warps, 64 threads)
        // Thread t copies tile rows t and t + 64 of every unit: the gathered
        // latent rows, as 16-byte cp.async into the swizzled K-major layout TMA
        // would write (zeros past the candidate count).  Up to c.gdepth tiles
        // are in flight per thread; a tile's full barrier gets one arrival per
        // warp once the warp's copies of it have landed.  Lane 0 of the first
        // warp also loads the query operand by TMA.
        constexpr int kRowsPerThread = kTileM / (32 * R::kProdWarps);
        const int t0 = (warp - R::kProdWarp0) * 32 + lane;
        const bool qloader = warp == R::kProdWarp0;
        if (qloader && lane == 0)
            tma_prefetch_desc(&tmB);
        const uint8_t *lat = static_cast<const uint8_t *>(p.latent);
        const int row_bytes = p.r * kEsz;
        const int pieces = c.nchunk * kPiecesPerChunk;
        const uint32_t a_base = smem_u32(smA);
        int stage = 0;
        uint32_t phase = 0;
        int pend = 0;
        int cur_bt = -1;
        int nb = 0;
        auto load_idx = [&](const Walk<kGather> &x, int row) -> int {
            const int slot = x.tile * kTileM + row;
            if (!x.ok() || slot >= p.n_gather)
                return -1;
            return __ldg(p.gather_idx + static_cast<int64_t>(seq_of(x.bt, p.T)) * p.L_out + slot);
        };
        auto signal_oldest = [&]() {
            int s_old = stage - pend;
            if (s_old < 0)
                s_old += c.stages;
            if (lane == 0)
                mbar_arrive(&full[s_old]);
            --pend;
        };
        Walk<kGather> w;
        w.init(p, u_begin, u_end, c.NT);
        int idx_next[kRowsPerThread];
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i)
            idx_next[i] = load_idx(w, t0 + 32 * R::kProdWarps * i);
        while (w.ok()) {
            Walk<kGather> wn = w;
            wn.next(p, c.NT);
            int idx[kRowsPerThread];
#pragma unroll
            for (int i = 0; i < kRowsPerThread; ++i) {
                idx[i] = idx_next[i];
                idx_next[i] = load_idx(wn, t0 + 32 * R::kProdWarps * i);   // one tile ahead
            }
            if (w.bt != cur_bt) {
                if (qloader && !load_query_operand(w.bt, nb))
                    break;
                cur_bt = w.bt;
                ++nb;
            }
            if (!warp_wait(&empty[stage], phase ^ 1u, abort_flag, p.status))
                break;
            const int b = seq_of(w.bt, p.T);
            const uint32_t dst0 = a_base + static_cast<uint32_t>(stage * c.a_stage_bytes);
#pragma unroll
            for (int i = 0; i < kRowsPerThread; ++i) {
                const int row = t0 + 32 * R::kProdWarps * i;
                const int slot = w.tile * kTileM + row;
                const bool in = slot < p.n_gather;
                const bool valid = in && idx[i] >= 0 && idx[i] < p.L_lat;
                if (in && !valid)
                    atomicCAS(p.status, 0, -7 /* LI_ERR_DEVICE_BOUNDS */);
                const uint8_t *src =
                    lat + (static_cast<int64_t>(b) * p.L_lat + (valid ? idx[i] : 0)) * row_bytes;
                const uint32_t nbytes = valid ? 16u : 0u;
                for (int j = 0; j < pieces; ++j) {
                    const int ch = j / kPiecesPerChunk;
                    const int qc = j % kPiecesPerChunk;
                    uint32_t off = static_cast<uint32_t>(row * kRowChunkBytes + qc * 16);
                    off ^= ((off >> 7) & (kFP8 ? 3u : 7u)) << 4;
                    cp_async_16(dst0 + static_cast<uint32_t>(ch * c.a_chunk_bytes) + off, src + j * 16,
                                nbytes);
                }
            }
            cp_async_commit();
            ++pend;
            if (++stage == c.stages) {
                stage = 0;
                phase ^= 1u;
            }
            if (pend > c.gdepth) {
                cp_async_wait_depth(c.gdepth);
                fence_proxy_async_smem();
                __syncwarp();
                signal_oldest();
            }
            w = wn;
        }
        // every copy this thread issued lands before the CTA can exit
        cp_async_wait_group<0>();
        fence_proxy_async_smem();
        __syncwarp();
        while (pend > 0)
            signal_oldest();
        if (qloader)
            drain_query_operand(nb);
        __syncwarp();
    } else if (warp >= R::kEpiWarp0) {
        griddep_wait();
        // ------------------------------------------------------------ epilogue
        constexpr int kCw = EpiShape<kH>::kCols;    // accumulator columns per warp
        const int e = warp - R::kEpiWarp0;
        const int quarter = warp & 3;               // TMEM lane quarter
        const int c0 = (e >> 2) * kCw;              // first accumulator column
        if (c0 < c.N) {
            // at H = 64 every warp owns one whole layer (N is a multiple of 64)
            const int ncols = kH == 64 ? kCw : min(kCw, c.N - c0);
            const int l0 = c0 / kH;                 // first layer (within the Gs scored)
            const int nlay = kH == 64 ? 1 : (ncols + kH - 1) / kH;
            const int row = quarter * 32 + lane;
            float *wq = misc->wq + e * kCw;
            float *sq = misc->sq + e * kCw;
            float *bq = misc->bq + e * kCw;
            const uint32_t tq = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                static_cast<uint32_t>(c0);
            // Per-token latent scale: in scan mode it arrived with the tile in
            // the stage's scale slot; gathering (HS followers) loads the
            // gathered token's scale one tile ahead, its index two tiles ahead.
            const bool stage_sc = !kGather && c.sc_stage;
            auto tok_of = [&](const Walk<kGather> &x) -> int {
                const int pos = x.tile * kTileM + row;
                if (!x.ok() || pos >= x.Lv)
                    return -1;
                if (kGather)
                    return __ldg(p.gather_idx + static_cast<int64_t>(seq_of(x.bt, p.T)) * p.L_out + pos);
                return pos;
            };
            auto scale_of = [&](const Walk<kGather> &x, int tok) -> float {
                if (p.lat_scale == nullptr)
                    return 1.f;
                if (tok < 0 || tok >= p.L_lat)
                    return 0.f;
                return __ldg(p.lat_scale + static_cast<int64_t>(seq_of(x.bt, p.T)) * p.L_lat + tok);
            };

            Walk<kGather> w;
            w.init(p, u_begin, u_end, c.NT);
            float sc_cur = stage_sc ? 0.f : scale_of(w, tok_of(w));
            float sc_next = 0.f;
            int tok1 = 0;                           // gather: token of the next unit
            if (kGather) {
                Walk<kGather> t = w;
                t.next(p, c.NT);
                tok1 = tok_of(t);
            }
            int acc = 0;
            uint32_t acc_phase = 0;
            int ord = 0;                            // tile ordinal within the CTA
            int est = 0;                            // the tile's stage (scales read in the stage)
            uint32_t est_phase = 0;
            int cur_bt = -1;
            float *out_row = p.scores;              // this thread's score row start (query row cur_bt)
            while (w.ok()) {
                int tok2 = 0;
                if (!stage_sc) {
                    // look ahead: the next unit's scale (its gathered index was
                    // loaded a tile ago) and, when gathering, the index after it
                    Walk<kGather> t = w;
                    t.next(p, c.NT);
                    sc_next = scale_of(t, kGather ? tok1 : tok_of(t));
                    if (kGather) {
                        t.next(p, c.NT);
                        tok2 = tok_of(t);
                    }
                }
                if (w.bt != cur_bt) {
                    __syncwarp();
                    const int64_t wrow = (w.bt * p.Gtot + p.g0) * p.H + c0;
                    for (int j = lane; j < ncols; j += 32) {
                        const float wv = p.w[wrow + j];
                        const float sv = p.q_abs_scale ? p.q_abs_scale[wrow + j] : 1.f;
                        if (kBeta) {
                            wq[j] = wv;
                            sq[j] = sv;
                            bq[j] = p.beta[wrow + j];
                        } else {
                            // the ReLU is taken as (x + |x|) / 2 (see below): the
                            // weight is halved
                            wq[j] = 0.5f * (wv * sv);
                        }
                    }
                    __syncwarp();
                    cur_bt = w.bt;
                    out_row = p.scores + (w.bt * (p.Gout ? p.Gout : Gs) + p.gout0 + l0) *
                                             static_cast<int64_t>(p.L_out) + row;
                }
                if (!warp_wait(&bars->tmem_full[acc], acc_phase, abort_flag, p.status))
                    break;
                tc_fence_after();
                const int pos = w.tile * kTileM + row;
                const bool valid = pos < w.Lv;
                float sc = sc_cur;
                if (stage_sc && c.sc_ring) {
                    // the tile's scales, in its ring slot (copied there by its MMA
                    // warp before the phase of tmem_full just waited for could
                    // complete); the read completes before the accumulator, and
                    // with it the slot, is released
                    sc = misc->scr[ord & (kScRing - 1)][row];
                    asm volatile("" ::"f"(sc));
                } else if (stage_sc) {
                    // the stage's copies have landed (their barrier completed before
                    // the MMAs ran); read this token's scale, then give the stage back
                    if (!warp_wait(&full[est], est_phase, abort_flag, p.status))
                        break;
                    sc = smS[est * kTileM + row];
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&empty[est]);
                    if (++est == c.stages) {
                        est = 0;
                        est_phase ^= 1u;
                    }
                }
                float *out = out_row + w.tile * kTileM;
                const uint32_t tacc = tq + static_cast<uint32_t>(acc * kAccStride);

                auto finish = [&](int lay, float u) {
                    if (!kBeta)
                        u *= sc;
                    if (valid && lay < nlay)
                        out[static_cast<int64_t>(lay) * p.L_out] = u;
                };
                // 32 accumulator columns starting at column `col` (relative to
                // c0) into the running sums (x, y)
                auto chunk = [&](const uint32_t(&v)[32], int col, float2 &x, float2 &y) {
                    if (kBeta) {
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            const float x0 = fmaf(__uint_as_float(v[j]) * sq[col + j], sc, bq[col + j]);
                            const float x1 = fmaf(__uint_as_float(v[j + 1]) * sq[col + j + 1], sc,
                                                  bq[col + j + 1]);
                            x = __ffma2_rn(make_float2(wq[col + j], wq[col + j + 1]),
                                           make_float2(fmaxf(x0, 0.f), fmaxf(x1, 0.f)), x);
                            if (kH == 16 && (j == 14 || j == 30)) {
                                finish((col + j) / 16, x.x + x.y);
                                x = make_float2(0.f, 0.f);
                            }
                        }
                    } else {
                        const float4 *w4 = reinterpret_cast<const float4 *>(wq + col);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 ww = w4[j];
                            // ReLU as x + |x| = 2 ReLU(x) in packed fp32 adds, against
                            // halved weights (both scalings by 2 are exact, so the sum
                            // is the same as with max(x, 0) and the full weight); two
                            // values per instruction instead of a max per value
                            const float c0 = __uint_as_float(v[4 * j]);
                            const float c1 = __uint_as_float(v[4 * j + 1]);
                            const float c2 = __uint_as_float(v[4 * j + 2]);
                            const float c3 = __uint_as_float(v[4 * j + 3]);
                            x = __ffma2_rn(make_float2(ww.x, ww.y),
                                           __fadd2_rn(make_float2(c0, c1), make_float2(fabsf(c0), fabsf(c1))), x);
                            y = __ffma2_rn(make_float2(ww.z, ww.w),
                                           __fadd2_rn(make_float2(c2, c3), make_float2(fabsf(c2), fabsf(c3))), y);
                            if (kH == 16 && (j == 3 || j == 7)) {
                                finish((col + 4 * j) / 16, (x.x + x.y) + (y.x + y.y));
                                x = make_float2(0.f, 0.f);
                                y = x;
                            }
                        }
                    }
                    if (kH == 32) {
                        finish(col / 32, (x.x + x.y) + (y.x + y.y));
                        x = make_float2(0.f, 0.f);
                        y = x;
                    }
                };
                // All of the warp's columns in flight at once; the accumulator is
                // released as soon as they have landed.
                uint32_t va[32], vb[32];
                if (ncols > 32)
                    tmem_ld64(tacc, va, vb);
                else
                    tmem_ld32(tacc, va);
                if constexpr (kCw > 64) {
                    uint32_t vc[32], vd[32];
                    if (ncols > 96)
                        tmem_ld64(tacc + 64u, vc, vd);
                    else if (ncols > 64)
                        tmem_ld32(tacc + 64u, vc);
                    tmem_ld_wait32(va);
                    tmem_regs_ready(vb);
                    tmem_regs_ready(vc);
                    tmem_regs_ready(vd);
                    // A relaxed arrival: a release would first wait for this warp's
                    // outstanding global loads and stores.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_relaxed(&bars->tmem_empty[acc]);
                    float2 x0 = make_float2(0.f, 0.f), y0 = x0, x1 = x0, y1 = x0;
                    chunk(va, 0, x0, y0);
                    if (ncols > 32)
                        chunk(vb, 32, x0, y0);
                    if (ncols > 64)
                        chunk(vc, 64, x1, y1);
                    if (ncols > 96)
                        chunk(vd, 96, x1, y1);
                    finish(0, ((x0.x + x0.y) + (y0.x + y0.y)) + ((x1.x + x1.y) + (y1.x + y1.y)));
                } else {
                    tmem_ld_wait32(va);
                    tmem_regs_ready(vb);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_relaxed(&bars->tmem_empty[acc]);
                    float2 x0 = make_float2(0.f, 0.f), y0 = x0;
                    chunk(va, 0, x0, y0);
                    if (ncols > 32)
                        chunk(vb, 32, x0, y0);
                    if (kH == 64)
                        finish(0, (x0.x + x0.y) + (y0.x + y0.y));
                }
                w.next(p, c.NT);
                sc_cur = sc_next;
                tok1 = tok2;
                ++ord;
                acc ^= 1;
                if (acc == 0)
                    acc_phase ^= 1u;
            }
        }
    }

    __syncthreads();
    if (warp == R::kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, static_cast<uint32_t>(kTmemCols));
    }
}

// ------------------------------------------------------------------ host side

// The latent's per-token fp32 scales are copied into each stage next to the
// tile (one 512-byte TMA box) in scan mode when the scale rows can be a TMA
// tensor: row stride L * 4 a multiple of 16 bytes.
bool scales_in_stage(const ScoreParams &p)
{
    return p.gather_idx == nullptr && p.lat_scale != nullptr && p.L_lat % 4 == 0;
}

bool make_config(const ScoreParams &p, bool fp8, TcConfig &c, int &smem_bytes)
{
    const int esz = fp8 ? 1 : 2;
    c.N = p.Gs * p.H;
    c.nchunk = p.r / kChunkElems;
    c.a_chunk_bytes = kTileM * kChunkElems * esz;
    c.b_chunk_bytes = c.N * kChunkElems * esz;
    c.a_stage_bytes = c.nchunk * c.a_chunk_bytes;
    c.b_bytes = c.nchunk * c.b_chunk_bytes;
    c.b_buf_stride = (c.b_bytes + 1023) & ~1023;
    c.sc_stage = scales_in_stage(p) ? 1 : 0;
    const int sc_bytes = c.sc_stage ? kTileM * 4 : 0;      // per stage
    const int bar_bytes = 2 * 8 * 8 + static_cast<int>(sizeof(Bars));
    const int fixed = 1024 /* alignment slack */ + ((bar_bytes + 15) & ~15) +
                      static_cast<int>(sizeof(Misc));
    // Two query-operand buffers when that still leaves >= 3 latent stages.
    int stages = (kSmemLimit - fixed - 2 * c.b_buf_stride) / (c.a_stage_bytes + sc_bytes);
    c.nbuf = 2;
    if (stages < 3) {
        c.nbuf = 1;
        stages = (kSmemLimit - fixed - c.b_buf_stride) / (c.a_stage_bytes + sc_bytes);
    }
    if (stages > 8)
        stages = 8;
    if (stages < 2)
        return false;
    c.stages = stages;
    // a shallow latent ring (the four-layer scan: two 48 KB query buffers
    // leave 4 stages) is not held up by the epilogue's reading of the scales
    c.sc_ring = c.sc_stage && stages < 6 ? 1 : 0;
    c.off_a = c.nbuf * c.b_buf_stride;
    c.off_sc = c.off_a + stages * c.a_stage_bytes;
    c.off_bar = c.off_sc + stages * sc_bytes;
    c.off_misc = (c.off_bar + 2 * stages * 8 + static_cast<int>(sizeof(Bars)) + 15) & ~15;
    smem_bytes = c.off_misc + static_cast<int>(sizeof(Misc)) + 1024;
    // one CTA per SM: a second CTA would only queue on the TMEM allocation
    if (smem_bytes < 116 * 1024)
        smem_bytes = 116 * 1024;
    c.cw = p.H == 128 ? 128 : 64;         // accumulator columns per epilogue warp (EpiShape)
    c.nepi = 4 * ((c.N + c.cw - 1) / c.cw);
    c.gdepth = stages - 1 < 3 ? stages - 1 : 3;
    const int Lrow = p.gather_idx ? p.L_out : p.L_lat;
    c.NT = (Lrow + kTileM - 1) / kTileM;
    c.U = static_cast<int64_t>(p.B) * p.T * c.NT;
    return smem_bytes <= kSmemLimit && c.nepi <= 4 * (256 / c.cw) && c.nepi * c.cw <= kConstCap;
}

template <bool kFP8, bool kGather, bool kBeta, int kH>
cudaError_t launch_t(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmS,
                     const ScoreParams &p,
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
                                             kSmemLimit);
        if (e != cudaSuccess)
            return e;
        set_bytes[dev].store(kSmemLimit, std::memory_order_relaxed);
    }
    int64_t grid = sm_count();
    if (grid > c.U)
        grid = c.U;
    if (grid <= 0)
        return cudaSuccess;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(Roles<kGather, kH>::kThreads),
                      static_cast<size_t>(smem_bytes), s, tmA, tmB, tmS, p, c);
}

template <bool kFP8, bool kGather, bool kBeta>
cudaError_t dispatch_h(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmS,
                       const ScoreParams &p,
                       const TcConfig &c, int smem_bytes, cudaStream_t s)
{
    switch (p.H) {
    case 16: return launch_t<kFP8, kGather, kBeta, 16>(tmA, tmB, tmS, p, c, smem_bytes, s);
    case 32: return launch_t<kFP8, kGather, kBeta, 32>(tmA, tmB, tmS, p, c, smem_bytes, s);
    case 64: return launch_t<kFP8, kGather, kBeta, 64>(tmA, tmB, tmS, p, c, smem_bytes, s);
    case 128: return launch_t<kFP8, kGather, kBeta, 128>(tmA, tmB, tmS, p, c, smem_bytes, s);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace

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

    CUtensorMap tmA, tmB, tmS;
    // latent [B][L][r] as a 4D map {64, L, r / 64, B} (element k of K chunk
    // ch of token t at t r + ch 64 + k); box {64, 128, r / 64, 1}: a tile's K
    // chunks land one after the other, each [128 rows][64 elements]
    {
        cuuint64_t dims[4] = {static_cast<cuuint64_t>(kChunkElems), static_cast<cuuint64_t>(p.L_lat),
                              static_cast<cuuint64_t>(p.r / kChunkElems), static_cast<cuuint64_t>(p.B)};
        cuuint64_t strides[3] = {static_cast<cuuint64_t>(p.r) * esz,
                                 static_cast<cuuint64_t>(kChunkElems) * esz,
                                 static_cast<cuuint64_t>(p.r) * esz * p.L_lat};
        cuuint32_t box[4] = {kChunkElems, kTileM, static_cast<cuuint32_t>(p.r / kChunkElems), 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (enc(&tmA, dt, 4, const_cast<void *>(p.latent), dims, strides, box, estr,
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
    // token scales [B][L] fp32 as a 2D map {L, B}; box {128, 1} (one tile's scales)
    memset(&tmS, 0, sizeof tmS);
    if (c.sc_stage) {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.L_lat), static_cast<cuuint64_t>(p.B)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.L_lat) * 4};
        cuuint32_t box[2] = {kTileM, 1};
        cuuint32_t estr[2] = {1, 1};
        if (enc(&tmS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(p.lat_scale), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const bool beta = p.beta != nullptr;
    if (fp8) {
        if (gather)
            return beta ? dispatch_h<true, true, true>(tmA, tmB, tmS, p, c, smem_bytes, s)
                        : dispatch_h<true, true, false>(tmA, tmB, tmS, p, c, smem_bytes, s);
        return beta ? dispatch_h<true, false, true>(tmA, tmB, tmS, p, c, smem_bytes, s)
                    : dispatch_h<true, false, false>(tmA, tmB, tmS, p, c, smem_bytes, s);
    }
    if (gather)
        return beta ? dispatch_h<false, true, true>(tmA, tmB, tmS, p, c, smem_bytes, s)
                    : dispatch_h<false, true, false>(tmA, tmB, tmS, p, c, smem_bytes, s);
    return beta ? dispatch_h<false, false, true>(tmA, tmB, tmS, p, c, smem_bytes, s)
                : dispatch_h<false, false, false>(tmA, tmB, tmS, p, c, smem_bytes, s);
}

} // namespace li
