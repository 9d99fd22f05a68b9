// Sparse MLA decode over the resolved rows ("Un contexte d'un million sur huit
// H200", section "Ce qui se passe": attention reads only the K selected
// latent rows).  Absorbed-MLA form: the 576-dim latent row is the key, its
// first 512 dims the value:
//   z = scale * q . row,  out = sum softmax(z) * row[:512],  lse = ln sum exp(z)
//
// General kernel (any head count that is a multiple of 8, both row formats):
// a CTA owns (query, 8 heads, a range of the K entries); each chunk of 32
// rows is dequantised to fp32 in shared memory; warp w is head w, lane l is
// row l for the scores and dims l + 32 i for the output; online softmax in
// the log2 domain.  With more than one range per query, partial
// (o, max, sum) records go to the pool's workspace and a combine kernel
// merges them.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "hs_internal.h"

namespace hs {
namespace {

constexpr int kHeadsPerCta = 8;
constexpr int kChunk = 32;
constexpr int kRowStride = kLatent + 1;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float e4m3_to_f32(uint8_t v) {
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)v, __NV_E4M3);
    return __half2float(__half(h));
}

struct AttnArgs {
    const __nv_bfloat16 *q;  // [rows][H][576]
    const int32_t *row_id;   // [rows][K]
    const uint8_t *pool;     // block pool base
    int layer, L, P, R, fmt, H, K, splits, kc, max_row;
    int32_t *err;
    float scale_log2;        // softmax_scale * log2(e)
    __nv_bfloat16 *out;      // [rows][H][512]
    float *lse;              // [rows][H] or null
    float *part;             // [rows][H][splits][514]
};

__global__ void __launch_bounds__(256) attn_simt_kernel(AttnArgs a) {
    extern __shared__ float smem[];
    float *qs = smem;                          // [8][576]
    float *rs = qs + kHeadsPerCta * kLatent;   // [32][577]
    __shared__ float valid[kChunk];
    const int row = blockIdx.x, hg = blockIdx.y, split = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = hg * kHeadsPerCta + warp;
    const int k0 = split * a.kc, k1 = min(a.K, k0 + a.kc);
    const __nv_bfloat16 *qrow = a.q + ((size_t)row * a.H + hg * kHeadsPerCta) * kLatent;
    for (int i = tid; i < kHeadsPerCta * kLatent; i += 256) qs[i] = __bfloat162float(qrow[i]);
    float o[16];
#pragma unroll
    for (int i = 0; i < 16; i++) o[i] = 0.f;
    float m = -INFINITY, l = 0.f;
    const int32_t *ids = a.row_id + (size_t)row * a.K;
    for (int c0 = k0; c0 < k1; c0 += kChunk) {
        __syncthreads();
        // dequantise up to 32 rows: each warp takes 4 rows
        for (int rr = warp; rr < kChunk; rr += 8) {
            const int k = c0 + rr;
            int32_t id = k < k1 ? ids[k] : -1;
            if (id >= a.max_row) {  // never read outside the pool
                if (lane == 0) set_error(a.err, HS_ERR_INDEX_RANGE);
                id = -1;
            }
            float *dst = rs + rr * kRowStride;
            if (lane == 0) valid[rr] = id >= 0 ? 1.f : 0.f;
            if (id < 0) {
                for (int i = lane; i < kLatent; i += 32) dst[i] = 0.f;
                continue;
            }
            const size_t blk = (size_t)(id / a.P), off = (size_t)(id % a.P);
            const uint8_t *src = a.pool + ((blk * a.L + a.layer) * a.P + off) * a.R;
            if (a.fmt == HS_ROW_E4M3_656) {
                const float *sc = (const float *)(src + 512);
                for (int i = lane; i < kNope; i += 32) dst[i] = e4m3_to_f32(src[i]) * sc[i >> 7];
                const __nv_bfloat16 *rope = (const __nv_bfloat16 *)(src + 528);
                for (int i = lane; i < kRope; i += 32) dst[kNope + i] = __bfloat162float(rope[i]);
            } else {
                const float *f = (const float *)src;
                for (int i = lane; i < kLatent; i += 32) dst[i] = f[i];
            }
        }
        __syncthreads();
        // scores: lane = row of the chunk
        const float *rrow = rs + lane * kRowStride;
        const float *qh = qs + warp * kLatent;
        float z = 0.f;
#pragma unroll 8
        for (int i = 0; i < kLatent; i++) z = fmaf(qh[i], rrow[i], z);
        z = valid[lane] > 0.f ? z * a.scale_log2 : -INFINITY;
        float cm = z;
#pragma unroll
        for (int ofs = 16; ofs > 0; ofs >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, ofs));
        const float mn = fmaxf(m, cm);
        if (mn == -INFINITY) continue;  // nothing valid yet (uniform over the warp)
        const float alpha = exp2f(m - mn);
        const float p = exp2f(z - mn);
        float ps = p;
#pragma unroll
        for (int ofs = 16; ofs > 0; ofs >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, ofs);
        l = l * alpha + ps;
        m = mn;
#pragma unroll
        for (int i = 0; i < 16; i++) o[i] *= alpha;
        for (int e = 0; e < kChunk; e++) {
            const float pe = __shfl_sync(0xffffffffu, p, e);
            const float *vr = rs + e * kRowStride + lane;
#pragma unroll
            for (int i = 0; i < 16; i++) o[i] = fmaf(pe, vr[32 * i], o[i]);
        }
    }
    if (a.splits == 1) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16 *dst = a.out + ((size_t)row * a.H + h) * kNope;
#pragma unroll
        for (int i = 0; i < 16; i++) dst[lane + 32 * i] = __float2bfloat16(o[i] * inv);
        if (a.lse && lane == 0)
            a.lse[(size_t)row * a.H + h] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    } else {
        float *dst = a.part + (((size_t)row * a.H + h) * a.splits + split) * (kNope + 2);
#pragma unroll
        for (int i = 0; i < 16; i++) dst[lane + 32 * i] = o[i];
        if (lane == 0) {
            dst[kNope] = m;
            dst[kNope + 1] = l;
        }
    }
}

__global__ void __launch_bounds__(128) attn_combine_kernel(const float *__restrict__ part, int splits,
                                                           __nv_bfloat16 *out, float *lse) {
    const size_t rh = blockIdx.x;  // row * H + h
    const float *p = part + rh * splits * (kNope + 2);
    float M = -INFINITY;
    for (int s = 0; s < splits; s++) M = fmaxf(M, p[s * (kNope + 2) + kNope]);
    float Lsum = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < splits; s++) {
        const float *ps = p + s * (kNope + 2);
        const float ms = ps[kNope], ls = ps[kNope + 1];
        if (ms == -INFINITY) continue;
        const float wgt = exp2f(ms - M);
        Lsum += ls * wgt;
#pragma unroll
        for (int i = 0; i < 4; i++) acc[i] += ps[threadIdx.x + 128 * i] * wgt;
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
#pragma unroll
    for (int i = 0; i < 4; i++) out[rh * kNope + threadIdx.x + 128 * i] = __float2bfloat16(acc[i] * inv);
    if (lse && threadIdx.x == 0) lse[rh] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
}

size_t simt_smem() { return ((size_t)kHeadsPerCta * kLatent + (size_t)kChunk * kRowStride) * 4; }

}  // namespace

int attention_splits(const hs_pool *p, int B, int nq) {
    const int rows = B * nq;
    const int ctas = rows * (p->cfg.mla_heads / kHeadsPerCta);
    int s = (2 * kNumSMs + ctas - 1) / ctas;
    s = s < 1 ? 1 : (s > kMaxSplits ? kMaxSplits : s);
    // at least one chunk of rows per split
    const int maxs = (p->cfg.top_k + kChunk - 1) / kChunk;
    return s > maxs ? maxs : s;
}

int attention_kernel_count(const hs_pool *p, int B, int nq) {
    const int K = p->cfg.top_k;
    int s = attention_splits(p, B, nq);
    const int kc = ((K + s - 1) / s + kChunk - 1) / kChunk * kChunk;
    s = (K + kc - 1) / kc;
    return s > 1 ? 2 : 1;
}

cudaError_t attention_setup(const hs_pool *p) {
    (void)p;
    return cudaFuncSetAttribute(attn_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)simt_smem());
}

cudaError_t launch_attention(const hs_pool *p, int layer, const void *q, const int32_t *row_id,
                             int B, int nq, float scale, void *out, float *lse, cudaStream_t st) {
    AttnArgs a;
    a.q = (const __nv_bfloat16 *)q;
    a.row_id = row_id;
    a.pool = p->d.rows;
    a.layer = layer;
    a.L = p->cfg.num_mla_layers;
    a.P = p->cfg.page_tokens;
    a.R = p->R;
    a.fmt = p->cfg.row_fmt;
    a.H = p->cfg.mla_heads;
    a.K = p->cfg.top_k;
    a.splits = attention_splits(p, B, nq);
    a.kc = ((a.K + a.splits - 1) / a.splits + kChunk - 1) / kChunk * kChunk;
    a.splits = (a.K + a.kc - 1) / a.kc;
    a.scale_log2 = scale * kLog2e;
    a.out = (__nv_bfloat16 *)out;
    a.lse = lse;
    a.part = p->d.attn_part;
    a.max_row = (int)(p->cfg.gpu_blocks * p->cfg.page_tokens);
    a.err = p->d.err;
    const int rows = B * nq;
    dim3 grid(rows, a.H / kHeadsPerCta, a.splits);
    attn_simt_kernel<<<grid, 256, simt_smem(), st>>>(a);
    if (a.splits > 1)
        attn_combine_kernel<<<rows * a.H, 128, 0, st>>>(p->d.attn_part, a.splits, a.out, lse);
    return cudaGetLastError();
}

cudaError_t indexer_setup(const hs_pool *p);
cudaError_t resolve_setup(const hs_pool *p);

cudaError_t setup_kernel_attributes(const hs_pool *p) {
    cudaError_t e = indexer_setup(p);
    if (e == cudaSuccess) e = resolve_setup(p);
    if (e == cudaSuccess) e = attention_setup(p);
    return e;
}

}  // namespace hs
