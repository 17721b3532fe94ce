// topk.cu -- exact per-row top-k by radix select.
//
// The TopK of eq. (8) in "LatentIndex: Cross-Layer Sharing with Layer-Specific
// Selection for Sparse Attention" (summary page, Methodology): each layer
// keeps the indices of its min(k, |V|) highest-scoring valid positions.
//
// Scores are mapped to order-preserving 32-bit keys (negative floats have all
// bits flipped, non-negative ones the sign bit set; -0 is first folded to +0
// so equal floats get equal keys).  The k-th largest key is found digit by
// digit, most significant first (12 + 12 + 8 bits), from shared-memory
// histograms; everything strictly above the threshold is emitted as soon as
// its digit decides it, and among keys equal to the threshold the lowest
// positions are taken (an in-order pass with block-wide ranks), which matches
// a full sort by (score desc, position asc).
//
// One 1024-thread CTA per row.  The row is read twice from global memory
// (histogram, then split); the elements in the threshold bin of the first
// digit are kept in shared memory when they fit, so the later digits cost no
// global traffic.  When they do not fit the row is re-read with a prefix
// filter instead -- the kernel needs no global scratch memory.
#include <atomic>
#include <cstdint>

#include "li_internal.cuh"

namespace li {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;
constexpr int kCap = 12288;

struct TopkSmem {
    uint32_t hist[kBins];
    uint32_t ckey[kCap];
    int32_t cpos[kCap];
    uint32_t warp_tot[kWarps];
    int emit_cnt;
    int cand_cnt;
    int sel_bin;
    uint32_t sel_gt;
    int running;
};

__device__ __forceinline__ uint32_t float_key(float x)
{
    if (x == 0.f)
        x = 0.f;                       // fold -0 into +0
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k)
{
    const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// Visit every valid element (pos, key) of a row: 16-byte loads when the row
// is 16-byte aligned, plain coalesced loads otherwise / for the tail.
template <class F>
__device__ __forceinline__ void for_row(const float *row, int V, F f)
{
    int head = 0;
    if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
        const int V4 = V & ~3;
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
        for (int i = threadIdx.x; 4 * i < V4; i += kThreads) {
            const float4 v = __ldg(r4 + i);
            f(4 * i, float_key(v.x));
            f(4 * i + 1, float_key(v.y));
            f(4 * i + 2, float_key(v.z));
            f(4 * i + 3, float_key(v.w));
        }
        head = V4;
    }
    for (int i = head + threadIdx.x; i < V; i += kThreads)
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
// strictly above it.  Thread t owns bins [4t, 4t+4).  All threads must call.
__device__ void select_bin(TopkSmem &sm, uint32_t need, int &bin, uint32_t &gt)
{
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        h[j] = sm.hist[4 * t + j];
    const uint32_t local = h[0] + h[1] + h[2] + h[3];
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
    for (int w2 = w + 1; w2 < kWarps; ++w2)
        above += sm.warp_tot[w2];
    uint32_t s = above;
#pragma unroll
    for (int j = 3; j >= 0; --j) {
        if (s < need && s + h[j] >= need) {
            sm.sel_bin = 4 * t + j;
            sm.sel_gt = s;
        }
        s += h[j];
    }
    __syncthreads();
    bin = sm.sel_bin;
    gt = sm.sel_gt;
    __syncthreads();
}

__device__ __forceinline__ void clear_hist(TopkSmem &sm)
{
    for (int i = threadIdx.x; i < kBins; i += kThreads)
        sm.hist[i] = 0u;
}

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const TopkParams p)
{
    extern __shared__ __align__(16) uint8_t smraw[];
    TopkSmem &sm = *reinterpret_cast<TopkSmem *>(smraw);
    const int tid = threadIdx.x;

    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
        const float *src = p.scores + row * p.in_stride;
        int V = p.L_row;
        if (p.valid_len != nullptr) {
            V = p.valid_len[row];
            V = V < 0 ? 0 : (V > p.L_row ? p.L_row : V);
        }
        const int64_t grp = row / p.rows_per_group;
        const int64_t orow = grp * p.group_stride + row % p.rows_per_group + p.row_offset;
        int32_t *oidx = p.idx + orow * p.k;
        float *oval = p.vals ? p.vals + orow * p.k : nullptr;
        const int32_t *map = p.map ? p.map + grp * p.map_stride : nullptr;
        const int nsel = p.k < V ? p.k : V;

        auto out_pos = [&](int pos) -> int32_t { return map ? map[pos] : pos; };
        auto emit = [&](bool pred, int pos, uint32_t key) {
            const int slot = reserve(&sm.emit_cnt, pred);
            if (pred && slot < p.k) {
                oidx[slot] = out_pos(pos);
                if (oval)
                    oval[slot] = key_float(key);
            }
        };

        // padding
        for (int j = nsel + tid; j < p.k; j += kThreads) {
            oidx[j] = -1;
            if (oval)
                oval[j] = -__int_as_float(0x7f800000);
        }
        if (nsel == V) {
            // everything valid is selected: positions in order
            for (int j = tid; j < V; j += kThreads) {
                oidx[j] = out_pos(j);
                if (oval)
                    oval[j] = src[j];
            }
            __syncthreads();
            continue;
        }

        // ---- digit 1: bits [31:20] over the whole row
        clear_hist(sm);
        if (tid == 0) {
            sm.emit_cnt = 0;
            sm.cand_cnt = 0;
            sm.running = 0;
        }
        __syncthreads();
        for_row(src, V, [&](int, uint32_t key) { atomicAdd(&sm.hist[key >> 20], 1u); });
        __syncthreads();
        int b1;
        uint32_t gt;
        select_bin(sm, static_cast<uint32_t>(nsel), b1, gt);
        uint32_t need = static_cast<uint32_t>(nsel) - gt;
        const bool store1 = sm.hist[b1] <= static_cast<uint32_t>(kCap);
        __syncthreads();
        clear_hist(sm);
        __syncthreads();

        // ---- split on digit 1; histogram digit 2 (bits [19:8]) of the bin
        for_row(src, V, [&](int pos, uint32_t key) {
            const int d1 = static_cast<int>(key >> 20);
            emit(d1 > b1, pos, key);
            const bool in = d1 == b1;
            if (in)
                atomicAdd(&sm.hist[(key >> 8) & 0xFFFu], 1u);
            if (store1) {
                const int slot = reserve(&sm.cand_cnt, in);
                if (in) {
                    sm.ckey[slot] = key;
                    sm.cpos[slot] = pos;
                }
            }
        });
        __syncthreads();
        int b2;
        select_bin(sm, need, b2, gt);
        need -= gt;
        const bool store2 = !store1 && sm.hist[b2] <= static_cast<uint32_t>(kCap);
        __syncthreads();
        clear_hist(sm);
        __syncthreads();

        // ---- split on digit 2; histogram digit 3 (bits [7:0])
        const uint32_t pre1 = static_cast<uint32_t>(b1) << 20;
        const uint32_t pre12 = pre1 | (static_cast<uint32_t>(b2) << 8);
        auto step3 = [&](int pos, uint32_t key) {
            const int d2 = static_cast<int>((key >> 8) & 0xFFFu);
            emit(d2 > b2, pos, key);
            const bool in = d2 == b2;
            if (in)
                atomicAdd(&sm.hist[key & 0xFFu], 1u);
            if (store2) {
                const int slot = reserve(&sm.cand_cnt, in);
                if (in) {
                    sm.ckey[slot] = key;
                    sm.cpos[slot] = pos;
                }
            }
        };
        const int n1 = sm.cand_cnt;
        if (store1) {
            for (int i = tid; i < n1; i += kThreads)
                step3(sm.cpos[i], sm.ckey[i]);
        } else {
            for_row(src, V, [&](int pos, uint32_t key) {
                if ((key & 0xFFF00000u) == pre1)
                    step3(pos, key);
            });
        }
        __syncthreads();
        int b3;
        select_bin(sm, need, b3, gt);
        need -= gt;                                  // ties needed at the threshold
        const uint32_t K = pre12 | static_cast<uint32_t>(b3);
        const bool take_all_ties = sm.hist[b3] == need;
        const int n2 = sm.cand_cnt;
        __syncthreads();

        // ---- emit keys above the threshold (and the ties when all are taken)
        auto step4 = [&](int pos, uint32_t key) {
            emit(key > K || (take_all_ties && key == K), pos, key);
        };
        if (store1) {
            for (int i = tid; i < n1; i += kThreads) {
                const uint32_t key = sm.ckey[i];
                if ((key & 0xFFFFFF00u) == pre12)
                    step4(sm.cpos[i], key);
            }
        } else if (store2) {
            for (int i = tid; i < n2; i += kThreads)
                step4(sm.cpos[i], sm.ckey[i]);
        } else {
            for_row(src, V, [&](int pos, uint32_t key) {
                if ((key & 0xFFFFFF00u) == pre12)
                    step4(pos, key);
            });
        }
        __syncthreads();

        // ---- ties: the `need` lowest positions whose key equals K, in order
        if (!take_all_ties) {
            for (int base = 0; base < V; base += kThreads) {
                const int pos = base + tid;
                const bool pred = pos < V && float_key(src[pos]) == K;
                const unsigned m = __ballot_sync(0xffffffffu, pred);
                const int lane = tid & 31, w = tid >> 5;
                if (lane == 0)
                    sm.warp_tot[w] = __popc(m);
                __syncthreads();
                uint32_t before = 0, total = 0;
                for (int w2 = 0; w2 < kWarps; ++w2) {
                    const uint32_t c = sm.warp_tot[w2];
                    before += w2 < w ? c : 0u;
                    total += c;
                }
                const uint32_t rank = static_cast<uint32_t>(sm.running) + before +
                                      __popc(m & ((1u << lane) - 1u));
                emit(pred && rank < need, pos, K);
                __syncthreads();
                if (tid == 0)
                    sm.running += static_cast<int>(total);
                __syncthreads();
                if (static_cast<uint32_t>(sm.running) >= need)
                    break;
            }
        }
        __syncthreads();
    }
}

} // namespace

cudaError_t launch_topk(const TopkParams &p, cudaStream_t s)
{
    if (p.rows <= 0)
        return cudaSuccess;
    constexpr int kMaxDev = 64;
    static std::atomic<int> attr_set[kMaxDev];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDev)
        dev = 0;
    const int smem = static_cast<int>(sizeof(TopkSmem));
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        attr_set[dev].store(1, std::memory_order_relaxed);
    }
    const int64_t grid = p.rows < 0x7FFFFFFF ? p.rows : 0x7FFFFFFF;
    topk_kernel<<<static_cast<unsigned>(grid), kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

} // namespace li
