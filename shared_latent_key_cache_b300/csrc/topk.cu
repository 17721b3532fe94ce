// topk.cu -- exact per-row top-k.
//
// The TopK of eq. (8) in "LatentIndex: Cross-Layer Sharing with Layer-Specific
// Selection for Sparse Attention" (summary page, Methodology): each layer
// keeps the indices of its min(k, |V|) highest-scoring valid positions.
//
// Scores are mapped to order-preserving 32-bit keys (negative floats have all
// bits flipped, non-negative ones the sign bit set; -0 is first folded to +0
// so equal floats get equal keys).  Selection is exact and matches a full
// sort by (score desc, position asc): among keys equal to the k-th largest
// the lowest positions are taken.
//
// Rows of at most 32,768 scores take the register-resident path below (one
// read of the row, three histogram levels over the keys held in registers).
// A few rows longer than 8,192 scores (all CTAs one per SM) are each spread
// over a thread-block cluster that merges its histograms in distributed
// shared memory (the cluster path, further below).
// Other long rows: one CTA per row, no global scratch memory (1024 threads;
// 512 threads and two CTAs per SM when there are at least two rows per SM):
//  1. Sampled thresholds (rows of >= 8192 valid scores selecting at most about
//     a quarter of them): 4096 stratified samples are histogrammed (12 + 12
//     key bits) to find two keys whose sample ranks sit five standard
//     deviations below (T_hi) and above (T_lo) k's expected rank.  One pass
//     over the row, 32 elements per thread in registers with block-wide
//     prefix sums for the output slots, emits every score >= T_hi (with
//     overwhelming probability all of them belong to the top-k) and copies the
//     band [T_lo, T_hi) into shared memory.  If the counts show that the k-th
//     score is not inside the band (or the band does not fit), step 2 runs
//     and overwrites every output slot.
//  2. Exact radix fallback: a histogram of the top 12 key bits over the row,
//     then a second pass that emits everything above the threshold bin and
//     copies the bin into shared memory (or, if it does not fit, re-reads the
//     row with a prefix filter for the lower digits).
//  3. Among the shared-memory candidates, the remaining need is resolved digit
//     by digit (12 + 12 + 8 bits) from shared-memory histograms; keys equal to
//     the final threshold are ranked by position (in shared memory, or by an
//     in-order pass over the row when there are very many of them).
#include <atomic>
#include <cstdint>

#include "li_internal.cuh"
#include "ptx.cuh"

namespace li {
namespace {

constexpr int kThreads = 1024;
constexpr int kBins = 4096;
constexpr int kCap = 16384;        // (key, position) candidates in shared memory (1024 threads)
constexpr int kTieCap = 2048;      // ties ranked in shared memory
constexpr int kSamples = 4096;     // 4 per thread
constexpr int kMinSampledRow = 8192;

// Shared memory of the long-row kernel with NT threads.  With 512 threads two
// CTAs share an SM, so the candidate list is half as long.
template <int NT>
struct TopkSmem {
    static constexpr int kNW = NT / 32;
    static constexpr int kCapN = NT == 1024 ? kCap : kCap / 2;
    uint32_t hist[kBins];
    uint32_t ckey[kCapN];
    int32_t cpos[kCapN];
    int32_t tpos[kTieCap];
    uint32_t warp_tot[kNW];
    int emit_cnt;
    int cand_cnt;
    int tie_cnt;
    int sel_bin;
    uint32_t sel_gt;
    int running;
    uint32_t tot_sure;
    uint32_t tot_band;
};

__device__ __forceinline__ uint32_t float_key(float x)
{
    // x + 0 folds -0 into +0 (IEEE round to nearest: -0 + +0 = +0); then
    // negatives have all bits flipped, non-negatives the sign bit set
    const uint32_t u = __float_as_uint(x + 0.f);
    return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k)
{
    const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// Visit every valid element (pos, key) of a row: 16-byte loads when the row
// is 16-byte aligned, plain coalesced loads otherwise / for the tail.
template <int NT, class F>
__device__ __forceinline__ void for_row(const float *row, int V, F f)
{
    int head = 0;
    if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
        const int V4 = V & ~3;
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
        for (int i = threadIdx.x; 4 * i < V4; i += NT) {
            const float4 v = __ldg(r4 + i);
            f(4 * i, float_key(v.x));
            f(4 * i + 1, float_key(v.y));
            f(4 * i + 2, float_key(v.z));
            f(4 * i + 3, float_key(v.w));
        }
        head = V4;
    }
    for (int i = head + threadIdx.x; i < V; i += NT)
        f(i, float_key(__ldg(row + i)));
}

// Warp-aggregated slot reservation on a shared counter for the calling lanes
// with pred set; returns this lane's slot (or -1).
__device__ __forceinline__ int reserve(int *counter, bool pred)
{
    const unsigned act = __activemask();
    const unsigned m = __ballot_sync(act, pred);
    if (m == 0u)
        return -1;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(m) - 1;
    int base = 0;
    if (lane == leader)
        base = atomicAdd(counter, __popc(m));
    base = __shfl_sync(act, base, leader);
    return pred ? base + __popc(m & ((1u << lane) - 1u)) : -1;
}

// Largest bin b with  sum_{d >= b} hist[d] >= need; returns b and the count
// strictly above it.  Thread t owns bins [B t, B t + B), B = 4096 / NT.  All
// threads must call.
template <int NT>
__device__ void select_bin(TopkSmem<NT> &sm, uint32_t need, int &bin, uint32_t &gt)
{
    constexpr int kB = kBins / NT;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    uint32_t h[kB];
    uint32_t local = 0;
#pragma unroll
    for (int j = 0; j < kB; ++j) {
        h[j] = sm.hist[kB * t + j];
        local += h[j];
    }
    uint32_t x = local;                       // inclusive suffix within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, x, off);
        if (lane + off < 32)
            x += y;
    }
    if (lane == 0)
        sm.warp_tot[w] = x;
    __syncthreads();
    uint32_t above = x - local;
    for (int w2 = w + 1; w2 < NT / 32; ++w2)
        above += sm.warp_tot[w2];
    uint32_t s = above;
#pragma unroll
    for (int j = kB - 1; j >= 0; --j) {
        if (s < need && s + h[j] >= need) {
            sm.sel_bin = kB * t + j;
            sm.sel_gt = s;
        }
        s += h[j];
    }
    __syncthreads();
    bin = sm.sel_bin;
    gt = sm.sel_gt;
    __syncthreads();
}

template <int NT>
__device__ __forceinline__ void clear_hist(TopkSmem<NT> &sm)
{
    for (int i = threadIdx.x; i < kBins; i += NT)
        sm.hist[i] = 0u;
}

// Exclusive prefix sum over the NT threads; *total gets the block sum.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(TopkSmem<NT> &sm, uint32_t v, uint32_t *total)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off)
            x += y;
    }
    if (lane == 31)
        sm.warp_tot[w] = x;
    __syncthreads();
    if (w == 0) {
        uint32_t y = lane < NT / 32 ? sm.warp_tot[lane] : 0u;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t z = __shfl_up_sync(0xffffffffu, y, off);
            if (lane >= off)
                y += z;
        }
        if (lane < NT / 32)
            sm.warp_tot[lane] = y;
    }
    __syncthreads();
    const uint32_t base = w > 0 ? sm.warp_tot[w - 1] : 0u;
    *total = sm.warp_tot[NT / 32 - 1];
    __syncthreads();
    return base + x - v;
}

// Digit d of a key: d = 0 -> bits [31:20], 1 -> [19:8], 2 -> [7:0].
__device__ __forceinline__ uint32_t digit(uint32_t key, int d)
{
    return d == 0 ? key >> 20 : (d == 1 ? (key >> 8) & 0xFFFu : key & 0xFFu);
}
__device__ __forceinline__ uint32_t digit_mask(int d)
{
    return d == 0 ? 0xFFF00000u : (d == 1 ? 0x000FFF00u : 0x000000FFu);
}
__device__ __forceinline__ int digit_shift(int d) { return d == 0 ? 20 : (d == 1 ? 8 : 0); }

struct RowOut {
    int32_t *idx;
    float *val;
    const int32_t *map;
    int k;
};

template <int NT>
__device__ __forceinline__ void emit(TopkSmem<NT> &sm, const RowOut &o, bool pred, int pos, uint32_t key)
{
    const int slot = reserve(&sm.emit_cnt, pred);
    if (pred && slot < o.k) {
        o.idx[slot] = o.map ? o.map[pos] : pos;
        if (o.val)
            o.val[slot] = key_float(key);
    }
}

// In-order pass over the row: emit the `need` lowest positions whose key is K.
template <int NT>
__device__ void tie_pass_global(TopkSmem<NT> &sm, const RowOut &o, const float *src, int V, uint32_t K,
                                uint32_t need)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0)
        sm.running = 0;
    __syncthreads();
    for (int base = 0; base < V; base += NT) {
        const int pos = base + tid;
        const bool pred = pos < V && float_key(src[pos]) == K;
        const unsigned m = __ballot_sync(0xffffffffu, pred);
        if (lane == 0)
            sm.warp_tot[w] = __popc(m);
        __syncthreads();
        uint32_t before = 0, total = 0;
        for (int w2 = 0; w2 < NT / 32; ++w2) {
            const uint32_t c = sm.warp_tot[w2];
            before += w2 < w ? c : 0u;
            total += c;
        }
        const uint32_t rank = static_cast<uint32_t>(sm.running) + before + __popc(m & ((1u << lane) - 1u));
        emit(sm, o, pred && rank < need, pos, K);
        __syncthreads();
        if (tid == 0)
            sm.running += static_cast<int>(total);
        __syncthreads();
        if (static_cast<uint32_t>(sm.running) >= need)
            break;
    }
    __syncthreads();
}

// Select the `need` largest keys among the n shared-memory candidates and emit
// them.  Returns true when done; false when the ties at the threshold are too
// many to rank in shared memory (then *Kout / *need_out describe the tie pass
// the caller runs over the row).
template <int NT>
__device__ bool select_candidates(TopkSmem<NT> &sm, const RowOut &o, int n, uint32_t need, uint32_t *Kout,
                                  uint32_t *need_out)
{
    const int tid = threadIdx.x;
    uint32_t prefix = 0, pmask = 0;
    uint32_t last_count = 0;
    for (int d = 0; d < 3; ++d) {
        clear_hist(sm);
        __syncthreads();
        for (int i = tid; i < n; i += NT) {
            const uint32_t key = sm.ckey[i];
            if ((key & pmask) == prefix)
                atomicAdd(&sm.hist[digit(key, d)], 1u);
        }
        __syncthreads();
        int b;
        uint32_t gt;
        select_bin(sm, need, b, gt);
        last_count = sm.hist[b];
        for (int i = tid; i < n; i += NT) {
            const uint32_t key = sm.ckey[i];
            const bool pred = (key & pmask) == prefix && digit(key, d) > static_cast<uint32_t>(b);
            emit(sm, o, pred, sm.cpos[i], key);
        }
        need -= gt;
        prefix |= static_cast<uint32_t>(b) << digit_shift(d);
        pmask |= digit_mask(d);
        __syncthreads();
    }
    const uint32_t K = prefix;           // the k-th largest key; `need` of its copies remain
    if (last_count == need) {
        for (int i = tid; i < n; i += NT)
            emit(sm, o, sm.ckey[i] == K, sm.cpos[i], K);
        __syncthreads();
        return true;
    }
    if (last_count > static_cast<uint32_t>(kTieCap)) {
        *Kout = K;
        *need_out = need;
        return false;
    }
    // rank the ties by position inside shared memory
    if (tid == 0)
        sm.tie_cnt = 0;
    __syncthreads();
    for (int i = tid; i < n; i += NT) {
        const bool pred = sm.ckey[i] == K;
        const int slot = reserve(&sm.tie_cnt, pred);
        if (pred)
            sm.tpos[slot] = sm.cpos[i];
    }
    __syncthreads();
    const int nt = sm.tie_cnt;
    for (int i = tid; i < nt; i += NT) {
        const int pi = sm.tpos[i];
        int rank = 0;
        for (int j = 0; j < nt; ++j)
            rank += sm.tpos[j] < pi ? 1 : 0;
        emit(sm, o, static_cast<uint32_t>(rank) < need, pi, K);
    }
    __syncthreads();
    return true;
}

// NT = 1024: one CTA per SM (few rows: each row's latency chain is what
// counts); NT = 512: two CTAs per SM, whose loads, barriers and scans overlap
// (many rows).
template <int NT>
__global__ void __launch_bounds__(NT, NT == 1024 ? 1 : 2) topk_kernel(const TopkParams p)
{
    constexpr int kCapN = TopkSmem<NT>::kCapN;
    extern __shared__ __align__(16) uint8_t smraw[];
    TopkSmem<NT> &sm = *reinterpret_cast<TopkSmem<NT> *>(smraw);
    const int tid = threadIdx.x;
    griddep_wait();
    griddep_launch_dependents();

    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
        const float *src = p.scores + row * p.in_stride;
        int V = p.L_row;
        if (p.valid_len != nullptr) {
            V = p.valid_len[row];
            V = V < 0 ? 0 : (V > p.L_row ? p.L_row : V);
        }
        const int64_t grp = row / p.rows_per_group;
        const int64_t orow = grp * p.group_stride + row % p.rows_per_group + p.row_offset;
        RowOut o;
        o.idx = p.idx + orow * p.k;
        o.val = p.vals ? p.vals + orow * (p.vals_stride ? p.vals_stride : p.k) : nullptr;
        o.map = p.map ? p.map + grp * p.map_stride : nullptr;
        o.k = p.k;
        const int nsel = p.k < V ? p.k : V;

        for (int j = nsel + tid; j < p.k; j += NT) {      // padding
            o.idx[j] = -1;
            if (o.val)
                o.val[j] = -__int_as_float(0x7f800000);
        }
        if (nsel == V) {
            // everything valid is selected: positions in order
            for (int j = tid; j < V; j += NT) {
                o.idx[j] = o.map ? o.map[j] : j;
                if (o.val)
                    o.val[j] = src[j];
            }
            __syncthreads();
            continue;
        }
        if (tid == 0) {
            sm.emit_cnt = 0;
            sm.cand_cnt = 0;
        }

        // ---------------------------------------------- 1. sampled thresholds
        bool have_cands = false;
        uint32_t need = static_cast<uint32_t>(nsel);
        const float pk = static_cast<float>(nsel) / static_cast<float>(V);
        const float sd = sqrtf(kSamples * pk * (1.f - pk));
        const float rlo_f = kSamples * pk + 5.f * sd + 2.f;
        const float rhi_f = kSamples * pk - 5.f * sd;
        if (V >= kMinSampledRow && rlo_f < 0.3f * kSamples) {
            clear_hist(sm);
            __syncthreads();
            for (int s2 = tid; s2 < kSamples; s2 += NT) {
                const int lo = static_cast<int>(static_cast<int64_t>(s2) * V / kSamples);
                const int hi = static_cast<int>(static_cast<int64_t>(s2 + 1) * V / kSamples);
                const int pos = lo + static_cast<int>(((static_cast<uint32_t>(s2) * 2654435761u) >> 8) %
                                                      static_cast<uint32_t>(hi - lo));
                const uint32_t key = float_key(__ldg(src + pos));
                sm.ckey[s2] = key;
                atomicAdd(&sm.hist[key >> 20], 1u);
            }
            __syncthreads();
            // sample key at a given (1-based, descending) rank, at 24-bit
            // precision: the low boundary of its (digit0, digit1) bin.
            // Expects the digit-0 histogram of the samples in sm.hist.
            auto sample_bin = [&](uint32_t rank) -> uint32_t {
                int c1, c2;
                uint32_t g1, g2;
                select_bin(sm, rank, c1, g1);
                clear_hist(sm);
                __syncthreads();
                for (int s2 = tid; s2 < kSamples; s2 += NT) {
                    const uint32_t key = sm.ckey[s2];
                    if ((key >> 20) == static_cast<uint32_t>(c1))
                        atomicAdd(&sm.hist[(key >> 8) & 0xFFFu], 1u);
                }
                __syncthreads();
                select_bin(sm, rank - g1, c2, g2);
                return (static_cast<uint32_t>(c1) << 20) | (static_cast<uint32_t>(c2) << 8);
            };
            const uint32_t T_lo = sample_bin(static_cast<uint32_t>(rlo_f));
            uint32_t T_hi = 0xFFFFFFFFu;              // no "certain" scores
            if (rhi_f >= 1.f) {
                clear_hist(sm);
                __syncthreads();
                for (int s2 = tid; s2 < kSamples; s2 += NT)
                    atomicAdd(&sm.hist[sm.ckey[s2] >> 20], 1u);
                __syncthreads();
                const uint32_t b = sample_bin(static_cast<uint32_t>(rhi_f));
                if (b < 0xFFFFFF00u)
                    T_hi = b + 0x100u;                // strictly above that bin
            }
            if (tid == 0) {
                sm.tot_sure = 0;
                sm.tot_band = 0;
            }
            __syncthreads();
            // one pass, 32 scores per thread per 32K chunk held in registers
            const bool al16 = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
            for (int base = 0; base < V; base += 32 * NT) {
                uint32_t key[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int pos = base + 4 * (tid + NT * i);
                    if (al16 && pos + 3 < V) {
                        const float4 v = __ldg(reinterpret_cast<const float4 *>(src + pos));
                        key[4 * i] = float_key(v.x);
                        key[4 * i + 1] = float_key(v.y);
                        key[4 * i + 2] = float_key(v.z);
                        key[4 * i + 3] = float_key(v.w);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            key[4 * i + j] = pos + j < V ? float_key(__ldg(src + pos + j)) : 0u;
                    }
                }
                uint32_t ns = 0, nb = 0;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int pos = base + 4 * (tid + NT * (e / 4)) + (e & 3);
                    const bool ok = pos < V;
                    ns += (ok && key[e] >= T_hi) ? 1u : 0u;
                    nb += (ok && key[e] >= T_lo && key[e] < T_hi) ? 1u : 0u;
                }
                uint32_t tot;
                const uint32_t off = block_excl_scan(sm, (ns << 16) | nb, &tot);
                uint32_t so = sm.tot_sure + (off >> 16);
                uint32_t bo = sm.tot_band + (off & 0xFFFFu);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int pos = base + 4 * (tid + NT * (e / 4)) + (e & 3);
                    if (pos >= V)
                        continue;
                    if (key[e] >= T_hi) {
                        if (so < static_cast<uint32_t>(nsel)) {
                            o.idx[so] = o.map ? o.map[pos] : pos;
                            if (o.val)
                                o.val[so] = key_float(key[e]);
                        }
                        ++so;
                    } else if (key[e] >= T_lo) {
                        if (bo < static_cast<uint32_t>(kCapN)) {
                            sm.ckey[bo] = key[e];
                            sm.cpos[bo] = pos;
                        }
                        ++bo;
                    }
                }
                __syncthreads();
                if (tid == 0) {
                    sm.tot_sure += tot >> 16;
                    sm.tot_band += tot & 0xFFFFu;
                }
                __syncthreads();
            }
            const uint32_t S = sm.tot_sure, Bn = sm.tot_band;
            have_cands = S < need && S + Bn >= need && Bn <= static_cast<uint32_t>(kCapN);
            if (have_cands) {
                need -= S;
                if (tid == 0) {
                    sm.emit_cnt = static_cast<int>(S);
                    sm.cand_cnt = static_cast<int>(Bn);
                }
            }
            __syncthreads();
        }

        int n = 0;
        bool stored = have_cands;
        int b1 = 0;
        if (have_cands) {
            n = sm.cand_cnt;
        } else {
            // ------------------------------------------ 2. exact radix fallback
            clear_hist(sm);
            if (tid == 0) {
                sm.emit_cnt = 0;
                sm.cand_cnt = 0;
            }
            __syncthreads();
            for_row<NT>(src, V, [&](int, uint32_t key) { atomicAdd(&sm.hist[key >> 20], 1u); });
            __syncthreads();
            uint32_t gt;
            select_bin(sm, need, b1, gt);
            stored = sm.hist[b1] <= static_cast<uint32_t>(kCapN);
            __syncthreads();
            for_row<NT>(src, V, [&](int pos, uint32_t key) {
                const uint32_t d1 = key >> 20;
                emit(sm, o, d1 > static_cast<uint32_t>(b1), pos, key);
                if (stored) {
                    const bool in = d1 == static_cast<uint32_t>(b1);
                    const int slot = reserve(&sm.cand_cnt, in);
                    if (in) {
                        sm.ckey[slot] = key;
                        sm.cpos[slot] = pos;
                    }
                }
            });
            __syncthreads();
            need -= gt;
            n = sm.cand_cnt;
            __syncthreads();
        }

        if (stored) {
            // --------------------------------- 3. select among the candidates
            uint32_t K = 0, need_eq = 0;
            if (!select_candidates(sm, o, n, need, &K, &need_eq))
                tie_pass_global(sm, o, src, V, K, need_eq);
        } else {
            // the threshold bin does not fit: lower digits by re-reading the row
            const uint32_t pre1 = static_cast<uint32_t>(b1) << 20;
            clear_hist(sm);
            __syncthreads();
            for_row<NT>(src, V, [&](int, uint32_t key) {
                if ((key & 0xFFF00000u) == pre1)
                    atomicAdd(&sm.hist[(key >> 8) & 0xFFFu], 1u);
            });
            __syncthreads();
            int b2;
            uint32_t gt;
            select_bin(sm, need, b2, gt);
            need -= gt;
            const uint32_t pre12 = pre1 | (static_cast<uint32_t>(b2) << 8);
            clear_hist(sm);
            __syncthreads();
            for_row<NT>(src, V, [&](int pos, uint32_t key) {
                const bool in = (key & 0xFFF00000u) == pre1;
                const uint32_t d2 = (key >> 8) & 0xFFFu;
                emit(sm, o, in && d2 > static_cast<uint32_t>(b2), pos, key);
                if (in && d2 == static_cast<uint32_t>(b2))
                    atomicAdd(&sm.hist[key & 0xFFu], 1u);
            });
            __syncthreads();
            int b3;
            select_bin(sm, need, b3, gt);
            need -= gt;
            const uint32_t K = pre12 | static_cast<uint32_t>(b3);
            const bool all_ties = sm.hist[b3] == need;
            __syncthreads();
            for_row<NT>(src, V, [&](int pos, uint32_t key) {
                const bool in = (key & 0xFFFFFF00u) == pre12;
                emit(sm, o, in && (key > K || (all_ties && key == K)), pos, key);
            });
            __syncthreads();
            if (!all_ties)
                tie_pass_global(sm, o, src, V, K, need);
        }
        __syncthreads();
    }
}


// ------------------------------------------------------------------------
// Register-resident path for rows of at most 32 * 1024 scores (the common
// decode case): each thread keeps its 32 keys in registers and the row is
// read from memory once.  The k-th largest key is found digit by digit with
// shared-memory histograms over the keys' offsets from the row minimum
// (11 + 11 + at most 10 bits; the first digit is chosen from the row's actual
// key range, so its 2048 bins resolve the distribution where it is), then
// every key above it is emitted and the ties at it are taken lowest position
// first (ranked by ordered block scans only when there are more of them than
// are needed).

constexpr int kRegPer = 32;
constexpr int kRegRow = kRegPer * kThreads;     // longest row: 32 keys x 1024 threads
constexpr int kRBins = 2048;

constexpr int kRCap = 4096;       // candidate list (keys in the threshold bin)
constexpr int kRankMax = 256;     // lists up to this long are ranked by counting

template <int NT>
struct RegSmem {
    static constexpr int kNW = NT / 32;
    uint32_t hist[kRBins];
    uint32_t ckey[kRCap];
    int32_t cpos[kRCap];
    uint32_t wa[kNW];
    uint32_t wb[kNW];
    uint32_t kmin, kmax;
    int sel_bin;
    uint32_t sel_gt;
    int slot;
    uint32_t out_cnt, cand_cnt;
    uint32_t scan_tot;        // block total of the last reg_excl_scan
};

// Largest bin b with  sum_{d >= b} hist[d] >= need; sets b and the count
// strictly above it.  Thread t owns bins [B t, B t + B), B = 2048 / NT; the
// suffix sums run as shuffles within warps and one shuffle scan of the warp
// totals in warp 0.  All threads must call.
template <int NT>
__device__ void reg_select_bin(RegSmem<NT> &sm, uint32_t need, int &bin, uint32_t &gt)
{
    constexpr int kB = kRBins / NT;
    constexpr int kNW = NT / 32;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    uint32_t h[kB];
    uint32_t local = 0;
#pragma unroll
    for (int j = 0; j < kB; ++j) {
        h[j] = sm.hist[kB * t + j];
        local += h[j];
    }
    uint32_t x = local;                       // inclusive suffix within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, x, off);
        if (lane + off < 32)
            x += y;
    }
    if (lane == 0)
        sm.wa[w] = x;
    __syncthreads();
    if (w == 0) {
        // exclusive suffix of the warp totals: keys in later warps' bins
        const uint32_t tot = lane < kNW ? sm.wa[lane] : 0u;
        uint32_t y = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t z = __shfl_down_sync(0xffffffffu, y, off);
            if (lane + off < 32)
                y += z;
        }
        if (lane < kNW)
            sm.wb[lane] = y - tot;
    }
    __syncthreads();
    uint32_t s = sm.wb[w] + (x - local);
#pragma unroll
    for (int j = kB - 1; j >= 0; --j) {
        if (s < need && s + h[j] >= need) {
            sm.sel_bin = kB * t + j;
            sm.sel_gt = s;
        }
        s += h[j];
    }
    __syncthreads();
    bin = sm.sel_bin;
    gt = sm.sel_gt;
    __syncthreads();
}

// Exclusive prefix sum of v over the block (thread order); *total = block
// sum.  Shuffles within warps, one shuffle scan of the warp totals in warp 0.
template <int NT>
__device__ __forceinline__ uint32_t reg_excl_scan(RegSmem<NT> &sm, uint32_t v, uint32_t *total)
{
    constexpr int kNW = NT / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off)
            x += y;
    }
    if (lane == 31)
        sm.wb[w] = x;
    __syncthreads();
    if (w == 0) {
        const uint32_t tot = lane < kNW ? sm.wb[lane] : 0u;
        uint32_t y = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t z = __shfl_up_sync(0xffffffffu, y, off);
            if (lane >= off)
                y += z;
        }
        if (lane < kNW)
            sm.wa[lane] = y - tot;            // exclusive base of warp `lane`
        if (lane == 31)
            sm.scan_tot = y;                  // block total
    }
    __syncthreads();
    const uint32_t base = sm.wa[w];
    *total = sm.scan_tot;
    __syncthreads();
    return base + x - v;
}

// kFull: the launch guarantees that every row holds exactly 32 NT valid
// scores (no valid lengths, no candidate list), so the passes carry no
// per-element validity test.
template <int NT, bool kFull>
__global__ void __launch_bounds__(NT, 1) topk_reg_kernel(const TopkParams p)
{
    constexpr int kNW = NT / 32;
    __shared__ RegSmem<NT> sm;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    griddep_wait();
    griddep_launch_dependents();

    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
        // A segmented row (p.segs > 1) is score row row / segs, positions
        // [s * seg_len, s * seg_len + Lr) with s = row % segs; its outputs are
        // positions in the whole row (pos_off added), valid_len is not used.
        int64_t rrow = row;
        int pos_off = 0;
        int Lr = p.L_row;
        if (p.segs > 1) {
            rrow = row / p.segs;
            pos_off = static_cast<int>(row % p.segs) * p.seg_len;
            Lr = min(p.seg_len, p.L_row - pos_off);
        }
        const float *src = p.scores + rrow * p.in_stride + pos_off;
        int V = Lr;
        if (p.valid_len != nullptr) {
            V = p.valid_len[row];
            V = V < 0 ? 0 : (V > Lr ? Lr : V);
        }
        const int64_t grp = row / p.rows_per_group;
        const int64_t orow = grp * p.group_stride + row % p.rows_per_group + p.row_offset;
        int32_t *oidx = p.idx + orow * p.k;
        float *oval = p.vals ? p.vals + orow * (p.vals_stride ? p.vals_stride : p.k) : nullptr;
        const int32_t *map = p.map ? p.map + grp * p.map_stride : nullptr;
        const int nsel = p.k < V ? p.k : V;
        // output index of row position pos (map and pos_off are never both used)
        auto gpos = [&](int pos) -> int { return map ? map[pos] : pos + pos_off; };

        for (int j = nsel + tid; j < p.k; j += NT) {      // padding
            oidx[j] = p.pad_idx;
            if (oval)
                oval[j] = -__int_as_float(0x7f800000);
        }
        if (nsel == V) {
            for (int j = tid; j < V; j += NT) {
                oidx[j] = gpos(j);
                if (oval)
                    oval[j] = src[j];
            }
            __syncthreads();
            continue;
        }

        // ---- load: element e of this thread is at position 4 (tid + NT (e / 4)) + e % 4
        uint32_t key[kRegPer];
        const bool al16 = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
        if (al16 && (Lr & 3) == 0) {
            // All eight 16-byte loads of the thread in flight at once: a load is
            // skipped only past the row's storage (Lr), positions in
            // [V, Lr) are read and then ignored through valid().
            const float4 *r4 = reinterpret_cast<const float4 *>(src);
            float4 v[kRegPer / 4];
#pragma unroll
            for (int i = 0; i < kRegPer / 4; ++i) {
                const int q = tid + NT * i;
                v[i] = 4 * q < Lr ? __ldg(r4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < kRegPer / 4; ++i) {
                key[4 * i] = float_key(v[i].x);
                key[4 * i + 1] = float_key(v[i].y);
                key[4 * i + 2] = float_key(v[i].z);
                key[4 * i + 3] = float_key(v[i].w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < kRegPer / 4; ++i) {
                const int pos = 4 * (tid + NT * i);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    key[4 * i + j] = pos + j < V ? float_key(__ldg(src + pos + j)) : 0u;
            }
        }
        const bool full = kFull || V == kRegPer * NT;
        auto valid = [&](int e) { return kFull || full || 4 * (tid + NT * (e >> 2)) + (e & 3) < V; };

        // ---- key range of the row
        uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
        for (int e = 0; e < kRegPer; ++e)
            if (valid(e)) {
                lo = min(lo, key[e]);
                hi = max(hi, key[e]);
            }
        lo = __reduce_min_sync(0xffffffffu, lo);
        hi = __reduce_max_sync(0xffffffffu, hi);
        if (lane == 0) {
            sm.wa[w] = lo;
            sm.wb[w] = hi;
        }
        __syncthreads();
        if (w == 0) {
            const uint32_t a = __reduce_min_sync(0xffffffffu, lane < kNW ? sm.wa[lane] : 0xFFFFFFFFu);
            const uint32_t b = __reduce_max_sync(0xffffffffu, lane < kNW ? sm.wb[lane] : 0u);
            if (lane == 0) {
                sm.kmin = a;
                sm.kmax = b;
                sm.slot = 0;
                sm.out_cnt = 0;
                sm.cand_cnt = 0;
            }
        }
        __syncthreads();
        const uint32_t kmin = sm.kmin;
        const uint32_t range = sm.kmax - kmin;
        const int nbits = range ? 32 - __clz(range) : 0;
        const int shift1 = nbits > 11 ? nbits - 11 : 0;
        const int shift2 = shift1 > 11 ? shift1 - 11 : 0;

        // ---- digits of the k-th largest offset (key - kmin)
        uint32_t need = static_cast<uint32_t>(nsel);
        uint32_t T = 0;          // offset of the threshold key
        uint32_t cnt_eq = 0;     // keys equal to it
        {
            // level 1: bits [shift1, nbits)
            for (int i = tid; i < kRBins; i += NT)
                sm.hist[i] = 0u;
            __syncthreads();
#pragma unroll
            for (int e = 0; e < kRegPer; ++e)
                if (valid(e))
                    atomicAdd(&sm.hist[(key[e] - kmin) >> shift1], 1u);
            __syncthreads();
            int b;
            uint32_t gt;
            reg_select_bin(sm, need, b, gt);
            cnt_eq = sm.hist[b];
            need -= gt;
            T = static_cast<uint32_t>(b) << shift1;
        }
        if (cnt_eq <= static_cast<uint32_t>(kRCap)) {
            // ---- usual case: keys above the level-1 bin are selected now, the
            // bin's keys move to a shared-memory list and the remaining digits
            // and the ties are resolved on that list only
            const uint32_t gt1 = static_cast<uint32_t>(nsel) - need;
            // offsets key - kmin inside the threshold bin: [lo_off, hi_off]
            // (T + 2^shift1 - 1 stays below 2^nbits, so it does not wrap)
            const uint32_t lo_off = T;
            const uint32_t hi_off = T + ((1u << shift1) - 1u);
            uint32_t n_sure = 0, n_cand = 0;
#pragma unroll
            for (int e = 0; e < kRegPer; ++e) {
                if (valid(e)) {
                    const uint32_t o = key[e] - kmin;
                    n_sure += o > hi_off ? 1u : 0u;
                    n_cand += o >= lo_off ? 1u : 0u;
                }
            }
            n_cand -= n_sure;
            // output slots by one block scan of (keys above, keys in the bin),
            // packed 16 + 16 bits (each count is at most 32,768)
            uint32_t both_tot = 0;
            const uint32_t both = reg_excl_scan(sm, (n_sure << 16) | n_cand, &both_tot);
            uint32_t so = both >> 16;
            uint32_t co = both & 0xFFFFu;
            if (map == nullptr && oval == nullptr) {
#pragma unroll
                for (int e = 0; e < kRegPer; ++e) {
                    const uint32_t o = key[e] - kmin;
                    if (valid(e) && o >= lo_off) {
                        const int pos = 4 * (tid + NT * (e >> 2)) + (e & 3);
                        if (o > hi_off) {
                            oidx[so] = pos + pos_off;
                            ++so;
                        } else {
                            sm.ckey[co] = key[e];
                            sm.cpos[co] = pos + pos_off;
                            ++co;
                        }
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < kRegPer; ++e) {
                    const uint32_t o = key[e] - kmin;
                    if (valid(e) && o >= lo_off) {
                        const int pos = 4 * (tid + NT * (e >> 2)) + (e & 3);
                        if (o > hi_off) {
                            oidx[so] = gpos(pos);
                            if (oval)
                                oval[so] = key_float(key[e]);
                            ++so;
                        } else {
                            sm.ckey[co] = key[e];
                            sm.cpos[co] = gpos(pos);
                            ++co;
                        }
                    }
                }
            }
            __syncthreads();
            const int n = static_cast<int>(cnt_eq);
            if (n <= kRankMax) {
                // Short list: each candidate's rank in (key desc, position asc)
                // order is the number of candidates ahead of it, counted by four
                // threads over a quarter of the list each; the `need` lowest
                // ranks are taken, rank r into output slot gt1 + r.
                const int part = tid & 3;
                const int per = (n + 3) >> 2;
                // NT / 4 candidates per round (one round at 1024 threads)
                for (int c0r = 0; c0r < n; c0r += NT / 4) {
                    const int c = c0r + (tid >> 2);
                    uint32_t ahead = 0, ck = 0;
                    int cp = 0;
                    if (c < n) {
                        ck = sm.ckey[c];
                        cp = sm.cpos[c];
                        const int j1 = min(n, (part + 1) * per);
                        for (int j = part * per; j < j1; ++j) {
                            const uint32_t kj = sm.ckey[j];
                            const int pj = sm.cpos[j];
                            ahead += (kj > ck || (kj == ck && pj < cp)) ? 1u : 0u;
                        }
                    }
                    ahead += __shfl_xor_sync(0xffffffffu, ahead, 1);
                    ahead += __shfl_xor_sync(0xffffffffu, ahead, 2);
                    if (c < n && part == 0 && ahead < need) {
                        const uint32_t sl = gt1 + ahead;
                        oidx[sl] = cp;
                        if (oval)
                            oval[sl] = key_float(ck);
                    }
                }
                __syncthreads();
                continue;
            }
            for (int level = 0; level < 2; ++level) {
                const int hs = level == 0 ? shift1 : shift2;
                const int ls = level == 0 ? shift2 : 0;
                if (hs == 0)
                    break;
                const uint32_t msk = (1u << (hs - ls)) - 1u;
                for (int i = tid; i < kRBins; i += NT)
                    sm.hist[i] = 0u;
                __syncthreads();
                for (int i = tid; i < n; i += NT) {
                    const uint32_t o = sm.ckey[i] - kmin;
                    if ((o >> hs) == (T >> hs))
                        atomicAdd(&sm.hist[(o >> ls) & msk], 1u);
                }
                __syncthreads();
                int b;
                uint32_t gt;
                reg_select_bin(sm, need, b, gt);
                cnt_eq = sm.hist[b];
                need -= gt;
                T |= static_cast<uint32_t>(b) << ls;
            }
            const uint32_t K = kmin + T;
            // list keys above K
            if (tid == 0)
                sm.slot = 0;
            __syncthreads();
            for (int i = tid; i < n; i += NT) {
                if (sm.ckey[i] > K) {
                    const uint32_t sl = gt1 + static_cast<uint32_t>(atomicAdd(&sm.slot, 1));
                    oidx[sl] = sm.cpos[i];
                    if (oval)
                        oval[sl] = key_float(sm.ckey[i]);
                }
            }
            __syncthreads();
            const uint32_t eq_base = gt1 + static_cast<uint32_t>(sm.slot);
            // ties at K: all, or the `need` lowest positions (radix select on positions)
            uint32_t pmax = 0xFFFFFFFFu;
            if (cnt_eq != need) {
                uint32_t P = 0, need_p = need;
                for (int lv = 0; lv < 3; ++lv) {
                    const int hs = lv == 0 ? 21 : (lv == 1 ? 10 : 0);
                    const int ws = lv == 2 ? 10 : 11;
                    const uint32_t pm = lv == 0 ? 0u : (0xFFFFFFFFu << (hs + ws));
                    for (int i = tid; i < kRBins; i += NT)
                        sm.hist[i] = 0u;
                    __syncthreads();
                    for (int i = tid; i < n; i += NT) {
                        const uint32_t up = static_cast<uint32_t>(sm.cpos[i]);
                        if (sm.ckey[i] == K && (up & pm) == (P & pm))
                            atomicAdd(&sm.hist[kRBins - 1 - ((up >> hs) & ((1u << ws) - 1u))], 1u);
                    }
                    __syncthreads();
                    // bins mirrored: the largest mirrored bin is the smallest digit
                    int b;
                    uint32_t gt;
                    reg_select_bin(sm, need_p, b, gt);
                    need_p -= gt;
                    P |= static_cast<uint32_t>(kRBins - 1 - b) << hs;
                }
                pmax = P;
            }
            if (tid == 0)
                sm.slot = 0;
            __syncthreads();
            for (int i = tid; i < n; i += NT) {
                const int pos = sm.cpos[i];
                if (sm.ckey[i] == K && static_cast<uint32_t>(pos) <= pmax) {
                    const uint32_t sl = eq_base + static_cast<uint32_t>(atomicAdd(&sm.slot, 1));
                    oidx[sl] = pos;
                    if (oval)
                        oval[sl] = key_float(K);
                }
            }
            __syncthreads();
            continue;
        }
        if (shift1 > 0) {
            // level 2: bits [shift2, shift1) of keys in the level-1 bin
            const uint32_t m2 = (1u << (shift1 - shift2)) - 1u;
            for (int i = tid; i < kRBins; i += NT)
                sm.hist[i] = 0u;
            __syncthreads();
#pragma unroll
            for (int e = 0; e < kRegPer; ++e) {
                const uint32_t o = key[e] - kmin;
                if (valid(e) && (o >> shift1) == (T >> shift1))
                    atomicAdd(&sm.hist[(o >> shift2) & m2], 1u);
            }
            __syncthreads();
            int b;
            uint32_t gt;
            reg_select_bin(sm, need, b, gt);
            cnt_eq = sm.hist[b];
            need -= gt;
            T |= static_cast<uint32_t>(b) << shift2;
        }
        if (shift2 > 0) {
            // level 3: bits [0, shift2) of keys matching the first two digits
            const uint32_t m3 = (1u << shift2) - 1u;
            for (int i = tid; i < kRBins; i += NT)
                sm.hist[i] = 0u;
            __syncthreads();
#pragma unroll
            for (int e = 0; e < kRegPer; ++e) {
                const uint32_t o = key[e] - kmin;
                if (valid(e) && (o >> shift2) == (T >> shift2))
                    atomicAdd(&sm.hist[o & m3], 1u);
            }
            __syncthreads();
            int b;
            uint32_t gt;
            reg_select_bin(sm, need, b, gt);
            cnt_eq = sm.hist[b];
            need -= gt;
            T |= static_cast<uint32_t>(b);
        }
        const uint32_t K = kmin + T;     // the k-th largest key; `need` of its cnt_eq copies are taken

        // ---- emit every key above K, positions in any order
        uint32_t mine = 0;
#pragma unroll
        for (int e = 0; e < kRegPer; ++e)
            mine += (valid(e) && key[e] > K) ? 1u : 0u;
        uint32_t sure = 0;
        uint32_t slot = reg_excl_scan(sm, mine, &sure);
#pragma unroll
        for (int e = 0; e < kRegPer; ++e) {
            if (valid(e) && key[e] > K) {
                const int pos = 4 * (tid + NT * (e >> 2)) + (e & 3);
                oidx[slot] = gpos(pos);
                if (oval)
                    oval[slot] = key_float(key[e]);
                ++slot;
            }
        }
        // ---- ties at K: all of them, or the `need` lowest positions
        if (cnt_eq == need) {
#pragma unroll
            for (int e = 0; e < kRegPer; ++e) {
                if (valid(e) && key[e] == K) {
                    const int pos = 4 * (tid + NT * (e >> 2)) + (e & 3);
                    const int s2 = static_cast<int>(sure) + atomicAdd(&sm.slot, 1);
                    oidx[s2] = gpos(pos);
                    if (oval)
                        oval[s2] = key_float(K);
                }
            }
        } else if (map != nullptr) {
            // positions of this row index a candidate list (map): ties are
            // taken by lowest mapped position, found by a radix select on
            // the mapped positions of the tied keys (the map's entries are
            // distinct), then emitted in any order
            uint32_t P = 0, need_p = need;
            for (int lv = 0; lv < 3; ++lv) {
                const int hs = lv == 0 ? 21 : (lv == 1 ? 10 : 0);
                const int ws = lv == 2 ? 10 : 11;
                const uint32_t pm = lv == 0 ? 0u : (0xFFFFFFFFu << (hs + ws));
                for (int i = tid; i < kRBins; i += NT)
                    sm.hist[i] = 0u;
                __syncthreads();
#pragma unroll
                for (int e = 0; e < kRegPer; ++e) {
                    if (valid(e) && key[e] == K) {
                        const uint32_t up = static_cast<uint32_t>(map[4 * (tid + NT * (e >> 2)) + (e & 3)]);
                        if ((up & pm) == (P & pm))
                            atomicAdd(&sm.hist[kRBins - 1 - ((up >> hs) & ((1u << ws) - 1u))], 1u);
                    }
                }
                __syncthreads();
                int b;
                uint32_t gt;
                reg_select_bin(sm, need_p, b, gt);
                need_p -= gt;
                P |= static_cast<uint32_t>(kRBins - 1 - b) << hs;
            }
            if (tid == 0)
                sm.slot = 0;
            __syncthreads();
#pragma unroll
            for (int e = 0; e < kRegPer; ++e) {
                if (valid(e) && key[e] == K) {
                    const int up = map[4 * (tid + NT * (e >> 2)) + (e & 3)];
                    if (static_cast<uint32_t>(up) <= P) {
                        const int s2 = static_cast<int>(sure) + atomicAdd(&sm.slot, 1);
                        oidx[s2] = up;
                        if (oval)
                            oval[s2] = key_float(K);
                    }
                }
            }
        } else {
            uint32_t run = 0;
#pragma unroll
            for (int i = 0; i < kRegPer / 4; ++i) {
                uint32_t c = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    c += (valid(4 * i + j) && key[4 * i + j] == K) ? 1u : 0u;
                uint32_t tot = 0;
                uint32_t r = run + reg_excl_scan(sm, c, &tot);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int e = 4 * i + j;
                    if (valid(e) && key[e] == K) {
                        if (r < need) {
                            const int pos = 4 * (tid + NT * i) + j;
                            oidx[sure + r] = gpos(pos);
                            if (oval)
                                oval[sure + r] = key_float(K);
                        }
                        ++r;
                    }
                }
                run += tot;
                if (run >= need)
                    break;          // uniform: every thread sees the same totals
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------------
// Cluster path for a few long rows (up to 16 x 32 x NT scores): one row is
// spread over a thread-block cluster, each CTA holding 32 keys per thread
// in registers, so that a handful of rows still occupies every SM.  The
// row's key histogram is merged level by level (key bits [21, 32), then
// [9, 21) inside the level-1 bin) in the first CTA's shared memory through
// distributed shared memory; the first CTA finds the threshold digit and
// writes it into every CTA.  Keys above the 23-bit threshold prefix are
// written by the CTA that holds them.  The few keys sharing the prefix are
// gathered in the first CTA and ranked there (key desc, position asc).  If
// there are many of them (near-equal scores), bits [0, 9) take a third
// merged level and the keys equal to the exact threshold are split between
// CTAs by position: every position of CTA c precedes those of CTA c + 1.

constexpr int kCB1 = 8192;       // level-1 bins: key bits [19, 32)
constexpr int kCB2 = 1024;       // level-2 bins: key bits [9, 19)
constexpr int kCB3 = 512;        // level-3 bins: key bits [0, 9)
constexpr int kCList = 256;      // prefix-sharing keys ranked in the first CTA
constexpr int kClusterMax = 16;

template <int NT>
struct ClusterSmem {
    static constexpr int kNW = NT / 32;
    uint32_t loc[kCB1];          // this CTA's histogram; first CTA: then the candidate list
    uint32_t m1[kCB1];           // merged histograms (first CTA)
    uint32_t m2[kCB2];
    uint32_t m3[kCB3];
    uint32_t tie[kClusterMax];   // keys equal to the threshold, per CTA (first CTA)
    uint32_t slot;               // output slots handed out (first CTA)
    uint32_t ncand;              // candidates listed (first CTA)
    uint32_t res[3];             // threshold digit, count above its bin, count in it
    uint32_t wa[kNW], wb[kNW];
    uint32_t scan_tot;
    uint32_t base_s, base_c;
    int sel_bin;
    uint32_t sel_gt;
};

__device__ __forceinline__ uint32_t cl_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cl_nrank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster: prior memory accesses are
// released to, and the peers' acquired from, the whole cluster.
__device__ __forceinline__ void cl_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cl_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cl_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cl_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of `local` (this CTA's shared memory) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cl_map(const void *local, uint32_t rank)
{
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
    return a;
}

__device__ __forceinline__ void cl_red_add(uint32_t addr, uint32_t v)
{
    asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t cl_atom_add(uint32_t addr, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.relaxed.cluster.shared::cluster.add.u32 %0, [%1], %2;"
                 : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void cl_st(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t cl_ld(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Largest bin b of hist[NB] with  sum_{d >= b} hist[d] >= need; sets b and
// the count strictly above it.  Thread t owns bins [B t, B t + B), B =
// NB / NT (one bin, or none past NB, when NB < NT).  All threads of the CTA
// must call.
template <int NT, int NB>
__device__ void cl_select_bin(ClusterSmem<NT> &sm, const uint32_t *hist, uint32_t need, int &bin,
                              uint32_t &gt)
{
    constexpr int kB = NB >= NT ? NB / NT : 1;
    constexpr int kNW = NT / 32;
    static_assert(NB >= NT ? NB % NT == 0 : NT % NB == 0, "bins per thread");
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    uint32_t h[kB];
    uint32_t local = 0;
#pragma unroll
    for (int j = 0; j < kB; ++j) {
        if constexpr (NB >= NT)
            h[j] = hist[kB * t + j];
        else
            h[j] = t < NB ? hist[t] : 0u;
        local += h[j];
    }
    uint32_t x = local;                       // inclusive suffix within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, x, off);
        if (lane + off < 32)
            x += y;
    }
    if (lane == 0)
        sm.wa[w] = x;
    __syncthreads();
    if (w == 0) {
        const uint32_t tot = lane < kNW ? sm.wa[lane] : 0u;
        uint32_t y = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t z = __shfl_down_sync(0xffffffffu, y, off);
            if (lane + off < 32)
                y += z;
        }
        if (lane < kNW)
            sm.wb[lane] = y - tot;
    }
    __syncthreads();
    uint32_t s = sm.wb[w] + (x - local);
#pragma unroll
    for (int j = kB - 1; j >= 0; --j) {
        if (s < need && s + h[j] >= need) {
            sm.sel_bin = kB * t + j;
            sm.sel_gt = s;
        }
        s += h[j];
    }
    __syncthreads();
    bin = sm.sel_bin;
    gt = sm.sel_gt;
}

// Exclusive prefix sum of v over the CTA in thread order; *total = CTA sum.
template <int NT>
__device__ __forceinline__ uint32_t cl_excl_scan(ClusterSmem<NT> &sm, uint32_t v, uint32_t *total)
{
    constexpr int kNW = NT / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off)
            x += y;
    }
    if (lane == 31)
        sm.wb[w] = x;
    __syncthreads();
    if (w == 0) {
        const uint32_t tot = lane < kNW ? sm.wb[lane] : 0u;
        uint32_t y = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t z = __shfl_up_sync(0xffffffffu, y, off);
            if (lane >= off)
                y += z;
        }
        if (lane < kNW)
            sm.wa[lane] = y - tot;
        if (lane == 31)
            sm.scan_tot = y;
    }
    __syncthreads();
    const uint32_t base = sm.wa[w];
    *total = sm.scan_tot;
    __syncthreads();
    return base + x - v;
}

// Adds this CTA's non-zero histogram bins loc[0, NB) into the first CTA's
// merged histogram `merged` (same offset in its shared memory).
template <int NT, int NB>
__device__ __forceinline__ void cl_push(const uint32_t *loc, const uint32_t *merged)
{
    const uint32_t m0 = cl_map(merged, 0);
    for (int i = threadIdx.x; i < NB; i += NT) {
        const uint32_t c = loc[i];
        if (c)
            cl_red_add(m0 + 4u * static_cast<uint32_t>(i), c);
    }
}

// In the first CTA: the threshold digit of the merged histogram `hist`,
// written into every CTA's res[] (the caller then synchronises the cluster).
template <int NT, int NB>
__device__ __forceinline__ void cl_broadcast_bin(ClusterSmem<NT> &sm, const uint32_t *hist,
                                                 uint32_t need, uint32_t ncta)
{
    int b;
    uint32_t gt;
    cl_select_bin<NT, NB>(sm, hist, need, b, gt);
    if (threadIdx.x < ncta) {
        const uint32_t r = cl_map(sm.res, threadIdx.x);
        cl_st(r, static_cast<uint32_t>(b));
        cl_st(r + 4u, gt);
        cl_st(r + 8u, hist[b]);
    }
}

// At most one CTA per SM runs (the path is taken only when rows x CTAs fit
// the SMs), so the registers are not capped for more.  NT = 256: 8K keys a
// CTA, up to 16 CTAs a row; NT = 1024: 32K keys a CTA (rows whose 256-thread
// clusters would not fit the SMs).
template <int NT>
__global__ void __launch_bounds__(NT, NT >= 1024 ? 1 : 2) topk_cluster_kernel(const TopkParams p)
{
    extern __shared__ __align__(16) uint8_t clraw[];
    ClusterSmem<NT> &sm = *reinterpret_cast<ClusterSmem<NT> *>(clraw);
    constexpr int kChunk = kRegPer * NT;
    const int tid = threadIdx.x;
    const uint32_t rank = cl_rank(), ncta = cl_nrank();
    const int64_t row = blockIdx.x / ncta;
    const int base = static_cast<int>(rank) * kChunk;
    griddep_wait();
    griddep_launch_dependents();

    const float *src = p.scores + row * p.in_stride;
    int V = p.L_row;
    if (p.valid_len != nullptr) {
        V = p.valid_len[row];
        V = V < 0 ? 0 : (V > p.L_row ? p.L_row : V);
    }
    const int64_t grp = row / p.rows_per_group;
    const int64_t orow = grp * p.group_stride + row % p.rows_per_group + p.row_offset;
    int32_t *oidx = p.idx + orow * p.k;
    float *oval = p.vals ? p.vals + orow * (p.vals_stride ? p.vals_stride : p.k) : nullptr;
    const int nsel = p.k < V ? p.k : V;
    if (rank == 0) {
        for (int j = nsel + tid; j < p.k; j += NT) {      // padding
            oidx[j] = p.pad_idx;
            if (oval)
                oval[j] = -__int_as_float(0x7f800000);
        }
    }
    if (nsel == V) {
        // every valid position is selected (no peer is touched: all CTAs of
        // the cluster take this branch and leave)
        const int end = min(V, base + kChunk);
        for (int j = base + tid; j < end; j += NT) {
            oidx[j] = j;
            if (oval)
                oval[j] = src[j];
        }
        return;
    }

    // ---- zero the merged histograms and counters (used in the first CTA)
    // and this CTA's level-1 histogram; the cluster barrier is completed
    // only before the first add into a peer
    if (rank == 0) {
        for (int i = tid; i < kCB1; i += NT)
            sm.m1[i] = 0u;
        for (int i = tid; i < kCB2; i += NT)
            sm.m2[i] = 0u;
        for (int i = tid; i < kCB3; i += NT)
            sm.m3[i] = 0u;
        if (tid < kClusterMax)
            sm.tie[tid] = 0u;
        if (tid == 0) {
            sm.slot = 0u;
            sm.ncand = 0u;
        }
    }
    for (int i = tid; i < kCB1; i += NT)
        sm.loc[i] = 0u;
    cl_arrive();

    // ---- load: element e of this thread is at position base + 4 (tid + NT (e / 4)) + e % 4
    uint32_t key[kRegPer];
    const float *csrc = src + base;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0 && (p.L_row & 3) == 0) {
        const float4 *r4 = reinterpret_cast<const float4 *>(csrc);
        const int lim = p.L_row - base;      // the row's storage past this chunk's start
        float4 v[kRegPer / 4];
#pragma unroll
        for (int i = 0; i < kRegPer / 4; ++i) {
            const int q = tid + NT * i;
            v[i] = 4 * q < lim ? __ldg(r4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kRegPer / 4; ++i) {
            key[4 * i] = float_key(v[i].x);
            key[4 * i + 1] = float_key(v[i].y);
            key[4 * i + 2] = float_key(v[i].z);
            key[4 * i + 3] = float_key(v[i].w);
        }
    } else {
#pragma unroll
        for (int i = 0; i < kRegPer / 4; ++i) {
            const int pos = base + 4 * (tid + NT * i);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                key[4 * i + j] = pos + j < V ? float_key(__ldg(src + pos + j)) : 0u;
        }
    }
    const bool full = base + kChunk <= V;
    auto posof = [&](int e) { return base + 4 * (tid + NT * (e >> 2)) + (e & 3); };
    auto valid = [&](int e) { return full || posof(e) < V; };

    // ---- level 1
    __syncthreads();
#pragma unroll
    for (int e = 0; e < kRegPer; ++e)
        if (valid(e))
            atomicAdd(&sm.loc[key[e] >> 19], 1u);
    __syncthreads();
    cl_wait();                                   // the first CTA's zeroing is done
    cl_push<NT, kCB1>(sm.loc, sm.m1);
    cl_sync();
    if (rank == 0)
        cl_broadcast_bin<NT, kCB1>(sm, sm.m1, static_cast<uint32_t>(nsel), ncta);
    cl_sync();
    const uint32_t b1 = sm.res[0];
    uint32_t need = static_cast<uint32_t>(nsel) - sm.res[1];
    uint32_t cnt = sm.res[2];

    uint32_t kge;              // keys >= kge are selected ...
    uint32_t keq = 0u;         // ... and, when tie_quota is set, keys == keq by position
    bool tie_quota = false;
    uint32_t quota = 0u;
    if (cnt == need) {
        kge = b1 << 19;
    } else {
        // ---- level 2: bits [9, 21) of the keys in the level-1 bin
        for (int i = tid; i < kCB2; i += NT)
            sm.loc[i] = 0u;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < kRegPer; ++e)
            if (valid(e) && (key[e] >> 19) == b1)
                atomicAdd(&sm.loc[(key[e] >> 9) & (kCB2 - 1)], 1u);
        __syncthreads();
        cl_push<NT, kCB2>(sm.loc, sm.m2);
        cl_sync();
        if (rank == 0)
            cl_broadcast_bin<NT, kCB2>(sm, sm.m2, need, ncta);
        cl_sync();
        const uint32_t t23 = (b1 << 10) | sm.res[0];
        need -= sm.res[1];
        cnt = sm.res[2];
        if (cnt == need) {
            kge = t23 << 9;
        } else if (cnt <= static_cast<uint32_t>(kCList)) {
            // ---- keys above the prefix are written here; those sharing it
            // are listed in the first CTA, which ranks them
            uint32_t ns = 0, nc = 0;
#pragma unroll
            for (int e = 0; e < kRegPer; ++e) {
                if (valid(e)) {
                    const uint32_t pk = key[e] >> 9;
                    ns += pk > t23 ? 1u : 0u;
                    nc += pk == t23 ? 1u : 0u;
                }
            }
            uint32_t tot = 0;
            const uint32_t both = cl_excl_scan(sm, (ns << 16) | nc, &tot);
            if (tid == 0) {
                sm.base_s = cl_atom_add(cl_map(&sm.slot, 0), tot >> 16);
                sm.base_c = cl_atom_add(cl_map(&sm.ncand, 0), tot & 0xFFFFu);
            }
            __syncthreads();
            uint32_t so = sm.base_s + (both >> 16);
            uint32_t co = sm.base_c + (both & 0xFFFFu);
            const uint32_t lk = cl_map(sm.loc, 0);
            const uint32_t lp = lk + 4u * kCList;
            // the list first: the barrier's release then waits for these few
            // shared-memory stores only, not for the output's global stores
#pragma unroll
            for (int e = 0; e < kRegPer; ++e) {
                if (valid(e) && (key[e] >> 9) == t23) {
                    cl_st(lk + 4u * co, key[e]);
                    cl_st(lp + 4u * co, static_cast<uint32_t>(posof(e)));
                    ++co;
                }
            }
            cl_sync();                           // list complete; no peer access after this
#pragma unroll
            for (int e = 0; e < kRegPer; ++e) {
                if (valid(e) && (key[e] >> 9) > t23) {
                    oidx[so] = posof(e);
                    if (oval)
                        oval[so] = key_float(key[e]);
                    ++so;
                }
            }
            if (rank == 0) {
                // rank of each listed key in (key desc, position asc) order
                const uint32_t first = static_cast<uint32_t>(nsel) - need;
                const int n = static_cast<int>(cnt);
                for (int c = tid; c < n; c += NT) {
                    const uint32_t ck = sm.loc[c];
                    const uint32_t cp = sm.loc[kCList + c];
                    uint32_t ahead = 0;
                    for (int j = 0; j < n; ++j) {
                        const uint32_t kj = sm.loc[j];
                        const uint32_t pj = sm.loc[kCList + j];
                        ahead += (kj > ck || (kj == ck && pj < cp)) ? 1u : 0u;
                    }
                    if (ahead < need) {
                        oidx[first + ahead] = static_cast<int>(cp);
                        if (oval)
                            oval[first + ahead] = key_float(ck);
                    }
                }
            }
            return;
        } else {
            // ---- level 3: bits [0, 9) of the keys sharing the prefix
            for (int i = tid; i < kCB3; i += NT)
                sm.loc[i] = 0u;
            __syncthreads();
#pragma unroll
            for (int e = 0; e < kRegPer; ++e)
                if (valid(e) && (key[e] >> 9) == t23)
                    atomicAdd(&sm.loc[key[e] & (kCB3 - 1)], 1u);
            __syncthreads();
            cl_push<NT, kCB3>(sm.loc, sm.m3);
            cl_sync();
            if (rank == 0)
                cl_broadcast_bin<NT, kCB3>(sm, sm.m3, need, ncta);
            cl_sync();
            const uint32_t K = (t23 << 9) | sm.res[0];
            need -= sm.res[1];
            cnt = sm.res[2];
            if (cnt == need) {
                kge = K;
            } else {
                // keys equal to K: the `need` lowest positions; CTA c takes
                // what remains of `need` after the ties of CTAs 0 .. c-1
                kge = K + 1u;                    // K is a finite score's key: no wrap
                keq = K;
                tie_quota = true;
                uint32_t mine = 0;
#pragma unroll
                for (int e = 0; e < kRegPer; ++e)
                    mine += (valid(e) && key[e] == K) ? 1u : 0u;
                uint32_t tot = 0;
                (void)cl_excl_scan(sm, mine, &tot);
                if (tid == 0)
                    cl_st(cl_map(&sm.tie[rank], 0), tot);
                cl_sync();
                uint32_t before = 0;
                if (tid == 0) {
                    const uint32_t t0 = cl_map(sm.tie, 0);
                    for (uint32_t r = 0; r < rank; ++r)
                        before += cl_ld(t0 + 4u * r);
                    sm.base_c = before;
                }
                __syncthreads();
                before = sm.base_c;
                quota = need > before ? min(need - before, tot) : 0u;
            }
        }
    }

    // ---- write every selected key; output slots from the first CTA's counter
    uint32_t take_tie = 0u;            // bit e: the tie in element e is taken
    if (tie_quota && quota > 0u) {
        uint32_t run = 0;
#pragma unroll
        for (int i = 0; i < kRegPer / 4; ++i) {
            uint32_t c = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                c += (valid(4 * i + j) && key[4 * i + j] == keq) ? 1u : 0u;
            uint32_t tot = 0;
            uint32_t r = run + cl_excl_scan(sm, c, &tot);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = 4 * i + j;
                if (valid(e) && key[e] == keq) {
                    if (r < quota)
                        take_tie |= 1u << e;
                    ++r;
                }
            }
            run += tot;
            if (run >= quota)
                break;              // uniform: every thread sees the same totals
        }
    }
    uint32_t mine = 0;
#pragma unroll
    for (int e = 0; e < kRegPer; ++e)
        mine += (valid(e) && (key[e] >= kge || ((take_tie >> e) & 1u))) ? 1u : 0u;
    uint32_t tot = 0;
    uint32_t so = cl_excl_scan(sm, mine, &tot);
    if (tid == 0)
        sm.base_s = cl_atom_add(cl_map(&sm.slot, 0), tot);
    __syncthreads();
    // the first CTA's slot counter is no longer accessed: a relaxed arrival
    // now (the atomic has returned), the wait before leaving, so the first
    // CTA outlives every access to its shared memory while no barrier waits
    // for the output's global stores
    cl_arrive_relaxed();
    so += sm.base_s;
#pragma unroll
    for (int e = 0; e < kRegPer; ++e) {
        if (valid(e) && (key[e] >= kge || ((take_tie >> e) & 1u))) {
            oidx[so] = posof(e);
            if (oval)
                oval[so] = key_float(key[e]);
            ++so;
        }
    }
    cl_wait();
}

} // namespace

namespace {

constexpr int kMaxDev = 64;
constexpr int kClusterNT = 256;
constexpr int kClusterChunk = kRegPer * kClusterNT;
constexpr int kClusterNTw = 1024;        // the wide cluster kernel
constexpr int kClusterChunkW = kRegPer * kClusterNTw;

int current_device()
{
    int dev = 0;
    cudaGetDevice(&dev);
    return dev < 0 || dev >= kMaxDev ? 0 : dev;
}

// Largest cluster the cluster path launches on this device: 16 when a
// cluster of 16 of its CTAs can be resident, else 8; -1 when its shared
// memory cannot be granted (the path is then not taken; 0 = not yet known).
int cluster_max(int dev)
{
    static std::atomic<int> cmax[kMaxDev];
    int c = cmax[dev].load(std::memory_order_relaxed);
    if (c != 0)
        return c;
    c = 8;
    if (cudaFuncSetAttribute(topk_cluster_kernel<kClusterNT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(ClusterSmem<kClusterNT>))) != cudaSuccess) {
        cudaGetLastError();
        cmax[dev].store(-1, std::memory_order_relaxed);      // the cluster path is not used
        return -1;
    }
    if (cudaFuncSetAttribute(topk_cluster_kernel<kClusterNT>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kClusterMax);
        cfg.blockDim = dim3(kClusterNT);
        cfg.dynamicSmemBytes = sizeof(ClusterSmem<kClusterNT>);
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = kClusterMax;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        cfg.attrs = a;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, topk_cluster_kernel<kClusterNT>, &cfg) == cudaSuccess &&
            n > 0)
            c = kClusterMax;
    }
    cudaGetLastError();
    cmax[dev].store(c, std::memory_order_relaxed);
    return c;
}

int sm_count(int dev)
{
    static std::atomic<int> sms[kMaxDev];
    int n = sms[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        sms[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// The wide cluster kernel's shared memory is granted on this device (set
// once).
bool wide_ready(int dev)
{
    static std::atomic<int> ok[kMaxDev];
    int v = ok[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        v = cudaFuncSetAttribute(topk_cluster_kernel<kClusterNTw>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sizeof(ClusterSmem<kClusterNTw>))) == cudaSuccess
                ? 1
                : -1;
        cudaGetLastError();
        ok[dev].store(v, std::memory_order_relaxed);
    }
    return v > 0;
}

struct ClusterShape {
    int ncta = 0;          // CTAs per row (0: another path)
    int nt = 0;            // threads per CTA
};

// The cluster path's shape for these rows.  It is taken when all its CTAs fit
// one per SM: each of its phases then runs on an otherwise idle SM.  256
// threads (8K keys) a CTA when those clusters fit (HS's anchor top-m: 8 rows
// of 128K -> 128 CTAs), else 1,024 threads (32K keys, clusters of 3-8) when
// those do (the per-layer top-k of 8 sequences x 4 layers at 128K: 32 rows
// -> 128 CTAs; 32.8 -> 30.6 us against the two-pass path).  With more CTAs than SMs (for example 128 rows of 32K) one
// CTA per row measured faster: every cluster phase costs a barrier and cold
// instruction fetches.
ClusterShape cluster_shape(const TopkParams &p)
{
    ClusterShape c;
    if (p.segs > 1 || p.map != nullptr || p.L_row <= kClusterChunk || p.rows <= 0)
        return c;
    const int dev = current_device();
    const int64_t sms = sm_count(dev);
    const int n256 = (p.L_row + kClusterChunk - 1) / kClusterChunk;
    if (n256 <= cluster_max(dev) && p.rows * n256 <= sms) {
        c.ncta = n256;
        c.nt = kClusterNT;
        return c;
    }
    const int nw = (p.L_row + kClusterChunkW - 1) / kClusterChunkW;
    // rows of at most 64K (two CTAs) measured no faster than the per-row paths
    if (nw >= 3 && nw <= 8 && p.rows * nw <= sms && wide_ready(dev)) {
        c.ncta = nw;
        c.nt = kClusterNTw;
    }
    return c;
}

template <int NT>
cudaError_t launch_topk_cluster(const TopkParams &p, int ncta, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.rows * ncta));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = sizeof(ClusterSmem<NT>);
    cfg.stream = s;
    cudaLaunchAttribute a[2];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = static_cast<unsigned>(ncta);
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    a[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = a;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, topk_cluster_kernel<NT>, p);
}

} // namespace

bool topk_cluster_path(const TopkParams &p) { return cluster_shape(p).ncta > 0; }

cudaError_t launch_topk(const TopkParams &p, cudaStream_t s)
{
    if (p.rows <= 0)
        return cudaSuccess;
    static std::atomic<int> attr_set[kMaxDev];
    const int dev = current_device();
    const ClusterShape cs = cluster_shape(p);
    if (cs.ncta > 0)
        return cs.nt == kClusterNT ? launch_topk_cluster<kClusterNT>(p, cs.ncta, s)
                                   : launch_topk_cluster<kClusterNTw>(p, cs.ncta, s);
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        cudaError_t e = cudaFuncSetAttribute(topk_kernel<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(sizeof(TopkSmem<1024>)));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(topk_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(sizeof(TopkSmem<512>)));
        if (e != cudaSuccess)
            return e;
        attr_set[dev].store(1, std::memory_order_relaxed);
    }
    const int64_t grid = p.rows < 0x7FFFFFFF ? p.rows : 0x7FFFFFFF;
    static_assert(kRegRow == kTopkRegRow, "register-resident row length");
    if (p.segs > 1 || p.L_row <= kRegRow) {
        // as many threads as the row needs at 32 keys each (at least 128).
        // Rows indexing a candidate list keep 1024 threads: every selected
        // key's output is a dependent load from the list, fewer per thread.
        const int Lr = p.map != nullptr ? kRegRow : (p.segs > 1 ? p.seg_len : p.L_row);
        // plain rows exactly as long as the threads' keys, indices only: the
        // variant without validity tests (for segments, candidate lists or
        // score outputs it measured slower: more live registers, more spills)
        const bool rows_full = p.map == nullptr && p.valid_len == nullptr && p.segs <= 1 &&
                               p.vals == nullptr;
        const dim3 g(static_cast<unsigned>(grid));
        if (Lr <= 32 * 128)
            return rows_full && Lr == 32 * 128 ? launch_pdl(topk_reg_kernel<128, true>, g, dim3(128), 0, s, p)
                                               : launch_pdl(topk_reg_kernel<128, false>, g, dim3(128), 0, s, p);
        if (Lr <= 32 * 256)
            return rows_full && Lr == 32 * 256 ? launch_pdl(topk_reg_kernel<256, true>, g, dim3(256), 0, s, p)
                                               : launch_pdl(topk_reg_kernel<256, false>, g, dim3(256), 0, s, p);
        if (Lr <= 32 * 512)
            return rows_full && Lr == 32 * 512 ? launch_pdl(topk_reg_kernel<512, true>, g, dim3(512), 0, s, p)
                                               : launch_pdl(topk_reg_kernel<512, false>, g, dim3(512), 0, s, p);
        return rows_full && Lr == 32 * 1024 ? launch_pdl(topk_reg_kernel<1024, true>, g, dim3(1024), 0, s, p)
                                            : launch_pdl(topk_reg_kernel<1024, false>, g, dim3(1024), 0, s, p);
    }
    // long rows: with at least two rows per SM, two 512-thread CTAs per SM
    if (p.rows >= 2 * static_cast<int64_t>(sm_count()))
        return launch_pdl(topk_kernel<512>, dim3(static_cast<unsigned>(grid)), dim3(512),
                          sizeof(TopkSmem<512>), s, p);
    return launch_pdl(topk_kernel<1024>, dim3(static_cast<unsigned>(grid)), dim3(1024), sizeof(TopkSmem<1024>),
                      s, p);
}

} // namespace li
