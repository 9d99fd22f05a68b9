// Token-partitioned decode on one GPU ("vLLM sert GLM-5.3 en contexte 1M sur
// 16 H200", section "Le mécanisme": decode context parallelism spreads a
// request's KV cache over the GPUs by tokens and gathers the fragments at
// every layer).  Here each shard selects its own candidates, the global top-K
// is taken over the union and the shards' attention partials are merged by
// their log-sum-exp.  Two kernels:
//
// dcp_merge_kernel, one CTA per row (request, query): the R partitions' local
//   top-K lists with their scores become candidates keyed by (score, lower
//   global token first); a bitonic sort in shared memory orders them, the K
//   best are the global top-K (every token of the global top-K is in its own
//   partition's local top-K, so the union is enough), written ascending by
//   token, and split back into each partition's local indices.
// dcp_combine_kernel, one CTA per (row, head): out = sum_r exp(lse_r - LSE) o_r
//   with LSE = log sum_r exp(lse_r); partitions without rows (lse = -inf)
//   weigh nothing.
#include <cuda_bf16.h>

#include "hs_internal.h"
#include "tc.cuh"

namespace {

constexpr int kMergeThreads = 1024;
constexpr int kMergeMax = 16384;  // R * K candidates per row

// Order-preserving key of an fp32 score.  -0 is first made +0: the two
// compare equal, so they must tie (and go to the lower token) like any other
// equal scores, not rank -0 below +0.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Bitonic sort of n (a power of two) 64-bit keys in shared memory, descending.
__device__ void bitonic_desc(unsigned long long *v, int n) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
                const int lo = 2 * i - (i & (stride - 1)), hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const unsigned long long a = v[lo], b = v[hi];
                if ((a < b) == desc) {
                    v[lo] = b;
                    v[hi] = a;
                }
            }
            __syncthreads();
        }
    }
}

// Ascending bitonic sort of n (a power of two) ints.
__device__ void bitonic_asc(int *v, int n) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
                const int lo = 2 * i - (i & (stride - 1)), hi = lo + stride;
                const bool asc = (lo & size) == 0;
                const int a = v[lo], b = v[hi];
                if ((a > b) == asc) {
                    v[lo] = b;
                    v[hi] = a;
                }
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(kMergeThreads) dcp_merge_kernel(
    const float *__restrict__ scores, int64_t stride, const int32_t *__restrict__ local,
    const int32_t *__restrict__ offsets, int R, int rows, int K, int ncand, int32_t *topk,
    int32_t *part_topk, int32_t *err) {
    extern __shared__ unsigned long long cand[];  // [ncand], then K ints
    int *sel = (int *)(cand + ncand);
    const int row = blockIdx.x;
    // candidate key: order-preserving score in the high word, the complement
    // of the global token in the low word (equal scores: lower token first);
    // 0 marks an empty candidate
    for (int i = threadIdx.x; i < ncand; i += blockDim.x) {
        unsigned long long key = 0;
        if (i < R * K) {
            const int r = i / K, k = i - r * K;
            const int32_t t = local[((size_t)r * rows + row) * K + k];
            if (t >= 0) {
                const int64_t g = (int64_t)offsets[r] + t;
                if (g < 0 || g >= 0x7fffffff) {
                    hs::set_error(err, HS_ERR_INDEX_RANGE);
                } else {
                    const float s = scores[((size_t)r * rows + row) * stride + t];
                    key = ((unsigned long long)order_key(s) << 32) | (uint32_t)(~(uint32_t)g);
                }
            }
        }
        cand[i] = key;
    }
    __syncthreads();
    bitonic_desc(cand, ncand);
    int kpow = 1;
    while (kpow < K) kpow <<= 1;
    // the K best, as global tokens (empty -> INT_MAX so they sort last)
    for (int i = threadIdx.x; i < kpow; i += blockDim.x) {
        const unsigned long long key = i < K ? cand[i] : 0ull;
        sel[i] = key ? (int)(~(uint32_t)(key & 0xffffffffu)) : 0x7fffffff;
    }
    __syncthreads();
    bitonic_asc(sel, kpow);
    int32_t *out = topk + (size_t)row * K;
    for (int i = threadIdx.x; i < K; i += blockDim.x) out[i] = sel[i] == 0x7fffffff ? -1 : sel[i];
    // per partition: its entries of the global top-K, as local indices (the
    // partitions are ascending token ranges, so each one's entries are one
    // contiguous run of the sorted list)
    for (int r = 0; r < R; r++) {
        const int lo = offsets[r], hi = r + 1 < R ? offsets[r + 1] : 0x7fffffff;
        int32_t *po = part_topk + ((size_t)r * rows + row) * K;
        // first entry >= lo by binary search (the list is ascending)
        int a = 0, b = K;
        while (a < b) {
            const int m = (a + b) >> 1;
            if (sel[m] < lo) a = m + 1; else b = m;
        }
        for (int i = threadIdx.x; i < K; i += blockDim.x) {
            const int j = a + i;
            po[i] = (j < K && sel[j] < hi && sel[j] != 0x7fffffff) ? sel[j] - lo : -1;
        }
    }
}

__global__ void __launch_bounds__(128) dcp_combine_kernel(const __nv_bfloat16 *__restrict__ o_parts,
                                                          const float *__restrict__ lse_parts, int R,
                                                          int rows, int H, __nv_bfloat16 *out,
                                                          float *lse) {
    const int rh = blockIdx.x;  // row * H + head
    const size_t plane = (size_t)rows * H;
    float m = -INFINITY;
    for (int r = 0; r < R; r++) m = fmaxf(m, lse_parts[r * plane + rh]);
    float wsum = 0.f;
    float w[8];  // R <= 8
    for (int r = 0; r < R; r++) {
        const float l = lse_parts[r * plane + rh];
        w[r] = (m == -INFINITY || l == -INFINITY) ? 0.f : __expf(l - m);
        wsum += w[r];
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    for (int d = threadIdx.x; d < hs::kNope; d += blockDim.x) {
        float acc = 0.f;
        for (int r = 0; r < R; r++)
            if (w[r] > 0.f) acc += w[r] * __bfloat162float(o_parts[(r * plane + rh) * hs::kNope + d]);
        out[(size_t)rh * hs::kNope + d] = __float2bfloat16(acc * inv);
    }
    if (threadIdx.x == 0 && lse) lse[rh] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

}  // namespace

namespace hs {
cudaError_t dcp_setup(const hs_pool *) {
    return cudaFuncSetAttribute(dcp_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kMergeMax * 8 + kMergeMax * 4);
}
}  // namespace hs

extern "C" {

hs_status hs_dcp_topk_merge(hs_pool *p, const float *scores, int64_t score_stride,
                            const int32_t *local_topk, const int32_t *offsets, int32_t R,
                            int32_t rows, int32_t *topk, int32_t *part_topk, cudaStream_t st) {
    if (!p || !scores || !local_topk || !offsets || !topk || !part_topk || R < 1 || R > 8 ||
        rows < 1 || score_stride < 1)
        return HS_ERR_INVALID_ARG;
    const int K = p->cfg.top_k;
    int ncand = 1;
    while (ncand < R * K) ncand <<= 1;
    int kpow = 1;
    while (kpow < K) kpow <<= 1;
    if (ncand > kMergeMax) return HS_ERR_CAPACITY;
    const size_t smem = (size_t)ncand * 8 + (size_t)kpow * 4;
    dcp_merge_kernel<<<rows, kMergeThreads, smem, st>>>(scores, score_stride, local_topk, offsets, R,
                                                        rows, K, ncand, topk, part_topk, p->d.err);
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

hs_status hs_dcp_combine(const void *o_parts, const float *lse_parts, int32_t R, int32_t rows,
                         int32_t H, void *out, float *lse, cudaStream_t st) {
    if (!o_parts || !lse_parts || !out || R < 1 || R > 8 || rows < 1 || H < 1)
        return HS_ERR_INVALID_ARG;
    dcp_combine_kernel<<<rows * H, 128, 0, st>>>((const __nv_bfloat16 *)o_parts, lse_parts, R, rows,
                                                  H, (__nv_bfloat16 *)out, lse);
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

}  // extern "C"
