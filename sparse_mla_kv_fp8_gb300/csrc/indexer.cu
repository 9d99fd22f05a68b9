// Indexer score ("Un contexte d'un million sur huit H200", section "Ce qui se
// passe": the indexer scores every cached token; its cache stays resident).
//
//   s[b][j][t] = sum_h w[b][j][h] * ReLU(sigma[b][t] * (q[b][j][h][:] . k[b][t][:]))
//
// General kernel: one CTA per 128-token tile of one request; the tile's keys
// and the request's queries are decoded to fp32 in shared memory; each thread
// owns one token and loops over (query, head).  Sums are fp32; with the
// synthetic inputs they are exact, so the result does not depend on order.
#include <cuda_fp8.h>

#include "hs_internal.h"

namespace hs {
namespace {

constexpr int kTile = 128;

__device__ __forceinline__ float e4m3_to_f32(uint8_t v) {
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)v, __NV_E4M3);
    return __half2float(__half(h));
}

template <int kFmt>  // 0 = E4M3 bytes, 1 = fp32
__global__ void __launch_bounds__(kTile) indexer_simt_kernel(
    const void *__restrict__ q, const float *__restrict__ w, const uint8_t *__restrict__ keys,
    const float *__restrict__ ksc, const int32_t *__restrict__ seq_len, int nq, int Hi, int Di,
    int maxT, float *__restrict__ scores, int64_t stride) {
    extern __shared__ float smem[];
    const int b = blockIdx.y;
    const int N = seq_len[b];
    const int t0 = blockIdx.x * kTile;
    if (t0 >= N) return;
    const int qn = nq * Hi * Di;
    float *qf = smem;                 // [nq*Hi*Di]
    float *wf = qf + qn;              // [nq*Hi]
    float *kt = wf + nq * Hi;         // [kTile][Di+1]
    const int ks = Di + 1;
    for (int i = threadIdx.x; i < qn; i += kTile) {
        if (kFmt == 0)
            qf[i] = e4m3_to_f32(((const uint8_t *)q)[(size_t)b * qn + i]);
        else
            qf[i] = ((const float *)q)[(size_t)b * qn + i];
    }
    for (int i = threadIdx.x; i < nq * Hi; i += kTile) wf[i] = w[(size_t)b * nq * Hi + i];
    const int ntok = min(kTile, N - t0);
    const size_t kbase = ((size_t)b * maxT + t0) * Di;
    for (int i = threadIdx.x; i < ntok * Di; i += kTile) {
        const int r = i / Di, d = i - r * Di;
        float v;
        if (kFmt == 0)
            v = e4m3_to_f32(keys[kbase + i]);
        else
            v = ((const float *)keys)[kbase + i];
        kt[r * ks + d] = v;
    }
    __syncthreads();
    const int r = threadIdx.x;
    if (r >= ntok) return;
    const int t = t0 + r;
    const float sig = ksc[(size_t)b * maxT + t];
    for (int j = 0; j < nq; j++) {
        float acc = 0.f;
        for (int h = 0; h < Hi; h++) {
            const float *qh = qf + (j * Hi + h) * Di;
            float dot = 0.f;
            for (int d = 0; d < Di; d++) dot = fmaf(qh[d], kt[r * ks + d], dot);
            const float x = sig * dot;
            acc = fmaf(wf[j * Hi + h], x > 0.f ? x : 0.f, acc);
        }
        scores[((size_t)b * nq + j) * stride + t] = acc;
    }
}

size_t simt_smem(const hs_pool *p, int nq) {
    const int Hi = p->cfg.idx_heads, Di = p->cfg.idx_dim;
    return ((size_t)nq * Hi * Di + nq * Hi + (size_t)kTile * (Di + 1)) * 4;
}

}  // namespace

cudaError_t indexer_setup(const hs_pool *p) {
    const size_t sm = simt_smem(p, p->nq_max);
    if (sm > 227 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(indexer_simt_kernel<0>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(indexer_simt_kernel<1>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
}

int indexer_kernel_count(const hs_pool *, int, int) { return 1; }

cudaError_t launch_indexer_score(const hs_pool *p, const void *q, const float *w, int B, int nq,
                                 float *scores, int64_t stride, cudaStream_t st) {
    const int maxT = p->cfg.max_tokens;
    dim3 grid((maxT + kTile - 1) / kTile, B);
    const size_t sm = simt_smem(p, nq);
    if (p->cfg.idx_fmt == HS_IDX_E4M3)
        indexer_simt_kernel<0><<<grid, kTile, sm, st>>>(q, w, p->d.idx_keys, p->d.idx_scale,
                                                         p->d.seq_len, nq, p->cfg.idx_heads,
                                                         p->cfg.idx_dim, maxT, scores, stride);
    else
        indexer_simt_kernel<1><<<grid, kTile, sm, st>>>(q, w, p->d.idx_keys, p->d.idx_scale,
                                                         p->d.seq_len, nq, p->cfg.idx_heads,
                                                         p->cfg.idx_dim, maxT, scores, stride);
    return cudaGetLastError();
}

}  // namespace hs
