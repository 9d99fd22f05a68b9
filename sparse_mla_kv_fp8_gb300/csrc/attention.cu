// Sparse MLA decode over the resolved rows ("Un contexte d'un million sur huit
// H200", section "Ce qui se passe": attention reads only the K selected
// latent rows).  Absorbed-MLA form: the 576-dim latent row is the key, its
// first 512 dims the value:
//   z = scale * q . row,  out = sum softmax(z) * row[:512],  lse = ln sum exp(z)
//
// Tensor-core kernel (E4M3 rows, head count a multiple of 64): one CTA owns
// one query, 64 heads and a range of the K entries, and computes in the
// transposed form so that both products are M=128 tcgen05 MMAs with fp16
// operands and fp32 accumulators in TMEM (fp16 rather than bf16: its 11-bit
// significand keeps the rounding of the dequantised rows, the queries and the
// probabilities about 8x smaller, which the output tolerance needs when a few
// rows dominate; magnitudes stay far inside fp16's range for scaled E4M3 rows):
//   S^T[row][head] = R[row][:576] . Q[head][:576]   M=128 rows,  N=64, K=576
//   O^T[dim][head] += R[row][dim] * P[row][head]    M=128 dims x4, N=64, K=128 rows
// TMEM: two S^T buffers (2 x 64 columns) + O^T (4 x 64 columns) + the
// softmax denominators (64 columns, from a ones x P^T MMA).  Warp 0 issues the
// MMAs, warp 1 owns TMEM, twelve worker warps dequantise the rows of each
// 128-row chunk (E4M3 x group scale -> fp16, in half2 with the scale split
// into two fp16s) straight into nine 16 KB K-blocks with the 128-byte
// swizzle; eight of them also run the softmax, and four (eight in a 2-CTA
// cluster) the epilogue.  The
// same K-blocks are the K-major A operand of S^T and the MN-major A operand
// of O^T, so each row is converted once.  Softmax warps (thread = row = TMEM
// lane) keep a per-head reference max in the log2 domain and rescale O^T
// only when a chunk raises a head's maximum by more than 2^8; P^T (fp16) is
// written over the rope K-block once S^T no longer needs it.  Per-K-block
// mbarriers let the conversion of chunk c+1 overlap the O^T MMAs of chunk c.
// Two row ranges of one query run as a 2-CTA cluster and merge through
// distributed shared memory.  Every wait is bounded.
//
// General kernel (any head count that is a multiple of 8, both row formats):
// a CTA owns (query, 8 heads, a range of the K entries); each chunk of 32
// rows is dequantised to fp32 in shared memory; warp w is head w, lane l is
// row l for the scores and dims l + 32 i for the output; online softmax in
// the log2 domain.  With more than one range per query, partial
// (o, max, sum) records go to the pool's workspace and a combine kernel
// merges them.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "tc.cuh"

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


// ------------------------------------------------------------------------
// tensor-core path
// ------------------------------------------------------------------------
constexpr int kTcRows = 128;         // rows per chunk (MMA M of S^T, K of O^T)
constexpr int kTcHeads = 64;         // heads per CTA (MMA N)
constexpr int kKBlocks = 9;          // 576 dims / 64
constexpr int kRBlock = kTcRows * 128;     // 16 KB: 128 rows x 64 fp16
constexpr int kQBlock = kTcHeads * 128;    // 8 KB: 64 heads x 64 fp16
constexpr int kWorkerWarps = 12;  // warps 2-13: rows, softmax, epilogue
constexpr int kAttnThreads = (2 + kWorkerWarps) * 32;
constexpr float kRescaleLog2 = 8.f;  // rescale O^T when a max grows by > 2^8

struct AttnTcSmem {
    static constexpr int r_off = 0;                              // 9 x 16 KB
    static constexpr int q_off = r_off + kKBlocks * kRBlock;     // 9 x 8 KB
    static constexpr int f_off = q_off + kKBlocks * kQBlock;     // floats
    static constexpr int nf = 64 * 3 + 4 * 64;                   // mref, lsum, alpha, red[4][64]
    static constexpr int ones_off = f_off + nf * 4;                // 128 x 16 fp16 ones
    static constexpr int bar_off = ones_off + 4096;
    static constexpr int nbar = 2 * kKBlocks + 2 + 2 + 6;
    static constexpr int tslot_off = bar_off + nbar * 8;
    static constexpr int bytes = tslot_off + 16 + 1024;          // + alignment slack
};
static_assert(AttnTcSmem::bytes <= 232448, "attention smem");

struct AttnTcArgs {
    const __nv_bfloat16 *q;  // [rows][H][576]
    const int32_t *row_id;   // [rows][K]
    const uint8_t *pool;
    int layer, L, P, H, K, splits, kc, max_row;
    float scale_log2;
    __nv_bfloat16 *out;      // [rows][H][512]
    float *lse;
    float *part;             // [rows][H][splits][514]
    int cluster;             // splits == 2 launched as 2-CTA clusters
    int q_ready;             // q may be read before waiting for the previous kernel
    int32_t *err;
};

__device__ __forceinline__ bool bar_or_softmax(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void bar_softmax() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// The softmax group: warps 2-5 (heads 0-31) and warps 6-9 (heads 32-63).
__device__ __forceinline__ bool bar_or_group(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 2, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void bar_group() { asm volatile("bar.sync 2, 256;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *(uint32_t *)&v;
}

// Two bf16 (low half first) -> two fp16, through fp32 (exact inside fp16's range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    return pack_f16(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Does any of eight bf16 values exceed fp16's range (|x| > 65504, which fp16
// rounds to infinity; NaN and infinity count too)?
__device__ __forceinline__ bool bf16x8_beyond_f16(uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 4; i++)
        bad |= (w[i] & 0x7FFFu) > 0x477Fu || ((w[i] >> 16) & 0x7FFFu) > 0x477Fu;
    return bad;
}

// Largest E4M3 magnitude times a group scale must stay inside fp16.
constexpr float kMaxF16 = 65504.f;
constexpr float kMaxE4M3 = 448.f;

__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
    return make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                      bf16x2_to_f16x2(v.w));
}

// An E4M3 pair times its group scale s, as fp16: the E4M3 values are exact in
// fp16 and s = s_hi + s_lo is split into two fp16s, so fma(x, s_hi, x * s_lo)
// rounds x * s once (up to the ~2^-18 of s that the split drops) in two
// half2 instructions instead of a widen / fp32 multiply / narrow per value.
// Below 2^-14 (fp16 subnormals) the split keeps s to 2^-25 absolute, so a
// value moves by at most 448 * 2^-25 (about 1.3e-5).
__device__ __forceinline__ uint32_t e4m3x2_scaled(__nv_fp8x2_storage_t v, __half2 s_hi, __half2 s_lo) {
    const __half2 x = __half2(__nv_cvt_fp8x2_to_halfraw2(v, __NV_E4M3));
    const __half2 y = __hfma2(x, s_hi, __hmul2(x, s_lo));
    return *(const uint32_t *)&y;
}

// 2^x with the hardware approximation (max 2 ulp); 2^-inf = +0.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kAttnThreads, 1) attn_tc_kernel(AttnTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *rb = smem + AttnTcSmem::r_off;
    uint8_t *qb = smem + AttnTcSmem::q_off;
    float *mref = (float *)(smem + AttnTcSmem::f_off);
    float *lsum = mref + 64;
    float *alpha = lsum + 64;
    float *red = alpha + 64;  // [4][64]
    uint8_t *ones = smem + AttnTcSmem::ones_off;
    uint64_t *kb_full = (uint64_t *)(smem + AttnTcSmem::bar_off);
    uint64_t *kb_empty = kb_full + kKBlocks;
    uint64_t *s_full = kb_empty + kKBlocks;
    uint64_t *s_empty = s_full + 2;
    uint64_t *p_full = s_empty + 2;
    uint64_t *o_done = p_full + 1;
    uint64_t *mma_done = o_done + 1;
    uint64_t *peer_ready = mma_done + 1;  // the peer split's row buffer is free
    uint64_t *peer_data = peer_ready + 1; // the peer split's partial has arrived
    uint64_t *q_full = peer_data + 1;     // the query blocks are in shared memory
    uint32_t *tslot = (uint32_t *)(smem + AttnTcSmem::tslot_off);

    const int qr = blockIdx.x, hh = blockIdx.y, split = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k0 = split * a.kc, k1 = min(a.K, k0 + a.kc);
    const int nchunks = (k1 - k0 + kTcRows - 1) / kTcRows;
    const int32_t *ids = a.row_id + (size_t)qr * a.K;

    if (threadIdx.x < 64) {
        mref[threadIdx.x] = -INFINITY;
        lsum[threadIdx.x] = 0.f;
    }
    for (int i = threadIdx.x; i < 4096 / 16; i += kAttnThreads)  // fp16 1.0 pairs
        ((uint4 *)ones)[i] = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kKBlocks; i++) {
            tc::mbar_init(&kb_full[i], kWorkerWarps);
            tc::mbar_init(&kb_empty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            tc::mbar_init(&s_full[i], 1);
            tc::mbar_init(&s_empty[i], 256);
        }
        tc::mbar_init(p_full, 256);
        tc::mbar_init(o_done, 1);
        tc::mbar_init(mma_done, 1);
        tc::mbar_init(peer_ready, 1);
        tc::mbar_init(peer_data, 256);
        tc::mbar_init(q_full, kWorkerWarps);
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tslot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (a.cluster) tc::cluster_sync();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    // everything above touched only this CTA's shared memory and TMEM: the
    // setup overlaps the previous kernel's tail; the next kernel may start too
    tc::grid_dep_launch();
    // Only the worker warps touch global memory; they wait for the previous
    // kernel below (after staging the queries when those were ready before it).
    const uint32_t s_col = 0;     // two S^T buffers: columns [0,64), [64,128)
    const uint32_t o_col = 128;   // O^T tiles: columns [128 + 64 g, ...)
    const uint32_t l_col = 384;   // per-row running sums of P: [384, 448)

    // Softmax of one chunk for heads [h_lo, h_lo + 32), run by 128 threads
    // (thread = chunk row = TMEM lane); the two 32-head halves together form a
    // 256-thread group.  Returns false (uniformly) when a wait ran out.  With
    // kLow the scores are re-read from TMEM 16 heads at a time instead of held
    // in 32 registers (the worker warps run it beside their own live state);
    // S^T(c) is then released at the end, which costs nothing because S^T(c+2)
    // cannot start before the row buffer has been refilled after PV(c+1).
    auto softmax_part = [&](int c, int h_lo, auto low) -> bool {
        constexpr bool kLow = decltype(low)::value;
        constexpr int kHeld = kLow ? 16 : 32;
        const int sp = warp & 3;
        const int r = sp * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(sp * 32) << 16);
        const int buf = c & 1;
        const int k = k0 + c * kTcRows + r;
        const int32_t id = k < k1 ? ids[k] : -1;
        const bool valid = id >= 0 && id < a.max_row;
        const bool w = tc::mbar_wait(&s_full[buf], (c >> 1) & 1, a.err);
        if (bar_or_group(!w)) return false;
        tc::fence_after_sync();
        const uint32_t sbase = lane_base + s_col + buf * kTcHeads + h_lo;
        float z[kHeld];
        auto load_scores = [&](int h0) {  // z <- scaled scores of heads h_lo+h0 ..
            tc::tmem_ld16(sbase + h0, z);
            if constexpr (!kLow) tc::tmem_ld16(sbase + h0 + 16, z + 16);
            tc::tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < kHeld; h++) z[h] = valid ? z[h] * a.scale_log2 : -INFINITY;
        };
        bool need = false;  // does any head's maximum grow by more than 2^8?
#pragma unroll
        for (int h0 = 0; h0 < 32; h0 += kHeld) {
            load_scores(h0);
#pragma unroll
            for (int h = 0; h < kHeld; h++) need |= z[h] > mref[h_lo + h0 + h] + kRescaleLog2;
        }
        if constexpr (!kLow) {
            tc::fence_before_sync();
            tc::mbar_arrive(&s_empty[buf]);  // S^T(c) is in registers
        }
        // kLow: z holds heads [16, 32) now; each later pass starts with the
        // half it holds and then loads the other
        int held = 32 - kHeld;
        if (bar_or_group(need)) {
            // chunk maximum of every head across the 128 rows
#pragma unroll
            for (int i = 0; i < 32 / kHeld; i++) {
                const int h0 = i == 0 ? held : 16 - held;
                if (i > 0) load_scores(h0);
#pragma unroll
                for (int h = 0; h < kHeld; h++) {
                    float m = z[h];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    if (lane == 0) red[sp * 64 + h_lo + h0 + h] = m;
                }
                if (i > 0) held = h0;
            }
            bar_group();
            if (r < 32) {
                const int hd = h_lo + r;
                const float cm = fmaxf(fmaxf(red[hd], red[64 + hd]), fmaxf(red[128 + hd], red[192 + hd]));
                const float mo = mref[hd];
                const float mn = fmaxf(mo, cm);
                alpha[hd] = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
                mref[hd] = mn;
            }
            bar_group();
            if (c > 0) {
                // O^T and l hold chunks < c: wait for them, then scale column h by alpha[h]
                const bool wo = tc::mbar_wait(o_done, (c - 1) & 1, a.err);
                if (bar_or_group(!wo)) return false;
                tc::fence_after_sync();
                for (int g = 0; g < 5; g++) {  // four O^T tiles, then the denominators
                    const uint32_t col = (g < 4 ? o_col + g * kTcHeads : l_col) + h_lo;
#pragma unroll
                    for (int h0 = 0; h0 < 32; h0 += 16) {
                        float ov[16];
                        const uint32_t ta = lane_base + col + h0;
                        tc::tmem_ld16(ta, ov);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; i++) ov[i] *= alpha[h_lo + h0 + i];
                        tc::tmem_st16(ta, ov);
                    }
                }
                tc::tmem_st_wait();
                tc::fence_before_sync();
            }
        }
        // P^T row r (fp16) -> the rope K-block (S^T(c) no longer reads it)
        uint8_t *prow = rb + 8 * kRBlock;
#pragma unroll
        for (int i = 0; i < 32 / kHeld; i++) {
            const int h0 = i == 0 ? held : 16 - held;
            if (i > 0) load_scores(h0);
#pragma unroll
            for (int c8 = 0; c8 < kHeld / 8; c8++) {
                const int hb = h_lo + h0 + c8 * 8;
                const float4 m0 = *(const float4 *)(mref + hb);
                const float4 m1 = *(const float4 *)(mref + hb + 4);
                const float mm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
                float pv[8];
#pragma unroll
                for (int e = 0; e < 8; e++)
                    pv[e] = (mm[e] == -INFINITY) ? 0.f : ex2_approx(z[c8 * 8 + e] - mm[e]);
                uint4 v;
                v.x = pack_f16(pv[0], pv[1]);
                v.y = pack_f16(pv[2], pv[3]);
                v.z = pack_f16(pv[4], pv[5]);
                v.w = pack_f16(pv[6], pv[7]);
                *(uint4 *)(prow + tc::sw128_offset(r, (hb >> 3))) = v;
            }
        }
        if constexpr (kLow) {
            tc::fence_before_sync();
            tc::mbar_arrive(&s_empty[buf]);  // done reading S^T(c)
        }
        tc::fence_async_smem();
        tc::mbar_arrive(p_full);
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            // every operand is fp16 (format 0 of kind::f16) in all three products
            const uint32_t idesc_s = tc::instr_desc(128, kTcHeads, 0, 0, 0, 0);
            const uint32_t idesc_o = tc::instr_desc(128, kTcHeads, 0, 0, 1, 1);
            const uint32_t idesc_l = tc::instr_desc(128, kTcHeads, 0, 0, 0, 1);
            const uint32_t ones_addr = tc::smem_addr(ones);
            const uint32_t r_addr = tc::smem_addr(rb), q_addr = tc::smem_addr(qb);
            const uint32_t p_addr = r_addr + 8 * kRBlock;
            bool ok = nchunks == 0 || tc::mbar_wait(q_full, 0, a.err);
            for (int c = 0; c < nchunks && ok; c++) {
                const int buf = c & 1;
                const uint32_t ph = c & 1;
                if (!(ok = tc::mbar_wait(&s_empty[buf], ((c >> 1) & 1) ^ 1, a.err))) break;
                for (int kb = 0; kb < kKBlocks && ok; kb++) {
                    if (!(ok = tc::mbar_wait(&kb_full[kb], ph, a.err))) break;
                    tc::fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < 4; kk++) {
                        const uint64_t ad = tc::smem_desc_sw128(r_addr + kb * kRBlock + kk * 32, 16, 1024);
                        const uint64_t bd = tc::smem_desc_sw128(q_addr + kb * kQBlock + kk * 32, 16, 1024);
                        tc::mma_f16(tmem + s_col + buf * kTcHeads, ad, bd, idesc_s, (kb | kk) != 0);
                    }
                }
                if (!ok) break;
                tc::mma_commit(&s_full[buf]);
                // O^T += V^T P^T once the softmax warps wrote P^T(c)
                if (!(ok = tc::mbar_wait(p_full, ph, a.err))) break;
                tc::fence_after_sync();
                for (int g = 0; g < 4; g++) {
#pragma unroll
                    for (int kk = 0; kk < 8; kk++) {
                        const uint64_t ad = tc::smem_desc_sw128(r_addr + 2 * g * kRBlock + kk * 2048, kRBlock, 1024);
                        const uint64_t bd = tc::smem_desc_sw128(p_addr + kk * 2048, kRBlock, 1024);
                        tc::mma_f16(tmem + o_col + g * kTcHeads, ad, bd, idesc_o, (c | kk) != 0);
                    }
                    tc::mma_commit(&kb_empty[2 * g]);
                    tc::mma_commit(&kb_empty[2 * g + 1]);
                }
                // softmax denominators: l[h] += sum_r P[r][h], as ones(128 x 128) P^T,
                // so every TMEM lane of the l columns holds the same sums
#pragma unroll
                for (int kk = 0; kk < 8; kk++) {
                    const uint64_t ad = tc::smem_desc(ones_addr, 128, 256, 0);
                    const uint64_t bd = tc::smem_desc_sw128(p_addr + kk * 2048, kRBlock, 1024);
                    tc::mma_f16(tmem + l_col, ad, bd, idesc_l, (c | kk) != 0);
                }
                tc::mma_commit(&kb_empty[8]);
                tc::mma_commit(o_done);
            }
            // every MMA issued by this thread has completed before TMEM is freed
            tc::mma_commit(mma_done);
            tc::mbar_wait(mma_done, 0, a.err);
        }
    } else if (warp >= 2) {
        // ------------------------------------------------------- row workers
        // Twelve warps convert each chunk.  A stage is one 128-dim scale group
        // (K-blocks 2g and 2g+1) or the rope block; its 1024 (row, 16-byte
        // slice) units are spread so that worker warp w holds rows 4w + 48u
        // .. 4w + 48u + 3 (u = 0, 1, and 2 for w < 8), 8 slices each.  Each
        // 8-lane group takes slices 0-3 or 4-7 of two adjacent rows, i.e. one
        // K-block: the 128-byte swizzle puts an even and an odd row's chunks
        // in disjoint bank slots, so the group's 16-byte stores are free of
        // bank conflicts (slices 0-3 and 4-7 of one row would land in two
        // K-blocks 16 KB apart, in the same slots); the rope stage swaps the
        // slice halves of odd rows for the same reason.  Loads run two
        // stages ahead of the conversion.  Warps 2-9 also run the softmax
        // (heads 0-31 on warps 2-5, 32-63 on warps 6-9) and warps 2-5 the
        // epilogue.
        const int wi = threadIdx.x - 64;  // 0..383
        const int c8 = (lane & 3) | (((lane >> 3) & 1) << 2);
        const int rw = (wi >> 5) * 4 + ((lane >> 4) & 1) * 2 + ((lane >> 2) & 1);  // row of u = 0
        const int c8r = c8 ^ ((rw & 1) << 2);  // rope slice
        const int nu = wi < 256 ? 3 : 2;
        auto id_at = [&](int c, int r) -> int32_t {
            const int k = k0 + c * kTcRows + r;
            return (c < nchunks && k < k1) ? ids[k] : -1;
        };
        // A row is addressed by its index in 656-byte units from the pool base
        // (below 2^32, which pool creation checks); ~0u marks a missing row.
        auto unit_of = [&](int32_t id) -> uint32_t {
            if (id >= a.max_row) {
                set_error(a.err, HS_ERR_INDEX_RANGE);
                id = -1;
            }
            if (id < 0) return ~0u;
            const uint32_t blk = (uint32_t)(id / a.P), off = (uint32_t)(id % a.P);
            return (blk * (uint32_t)a.L + (uint32_t)a.layer) * (uint32_t)a.P + off;
        };
        const uint4 z = make_uint4(0, 0, 0, 0);
        // stage st of row unit ru: 16 bytes of slice c8 (c8r for the rope) and
        // (st < 4) its scale
        auto ld_stage = [&](uint32_t ru, int st, uint4 &d, uint32_t &sc) {
            if (ru == ~0u) {
                d = z;
                sc = 0;
                return;
            }
            const uint8_t *row = a.pool + (size_t)ru * 656;
            d = tc::ld_nc16(row + (st < 4 ? 128 * st + 16 * c8 : 528 + 16 * c8r));
            sc = st < 4 ? tc::ld_nc4(row + 512 + 4 * st) : 0u;
        };
        uint32_t ru[3];
        uint4 d0[3], d1[3];
        uint32_t f0[3], f1[3];
        int32_t idn[3];  // the next chunk's row ids load while this chunk converts
        auto issue_first = [&]() {  // row units and stage 0 of the chunk in idn
#pragma unroll
            for (int u = 0; u < 3; u++) {
                ru[u] = unit_of(idn[u]);
                ld_stage(ru[u], 0, d0[u], f0[u]);
            }
        };
        // this CTA's 64 query heads -> nine K-major 128-byte-swizzled blocks
        const uint8_t *qsrc = (const uint8_t *)(a.q + ((size_t)qr * a.H + hh * kTcHeads) * kLatent);
        uint4 qv[12];
        auto q_load = [&]() {
#pragma unroll
            for (int j = 0; j < 12; j++) {  // 64 heads x 72 slices of 16 B
                const int i = wi + 384 * j, h = i / 72, c16 = i - h * 72;
                qv[j] = tc::ld_nc16(qsrc + (size_t)h * (kLatent * 2) + c16 * 16);
            }
        };
        bool range_bad = false;  // a value beyond fp16's range (reported once at the end)
        auto q_store = [&]() {
#pragma unroll
            for (int j = 0; j < 12; j++) {
                const int i = wi + 384 * j, h = i / 72, c16 = i - h * 72;
                range_bad |= bf16x8_beyond_f16(qv[j]);
                *(uint4 *)(qb + (c16 >> 3) * kQBlock + tc::sw128_offset(h, c16 & 7)) = bf16x8_to_f16x8(qv[j]);
            }
            tc::fence_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(q_full);
        };
        if (a.q_ready) {  // the queries overlap the previous kernel's tail
            q_load();
            q_store();
        }
        tc::grid_dep_wait();  // the row ids come from the previous kernel
#pragma unroll
        for (int u = 0; u < 3; u++) idn[u] = u < nu ? id_at(0, rw + 48 * u) : -1;
        if (a.q_ready) {
            issue_first();
        } else {  // the queries are staged while the first rows are in flight
            q_load();
            issue_first();
            q_store();
        }
        bool ok = true;
        for (int c = 0; c < nchunks; c++) {
#pragma unroll
            for (int u = 0; u < 3; u++) idn[u] = u < nu ? id_at(c + 1, rw + 48 * u) : -1;
            if (ok) {
#pragma unroll
                for (int st = 0; st < 5; st++) {
                    if (st == 0) {
#pragma unroll
                        for (int u = 0; u < 3; u++) ld_stage(ru[u], 1, d1[u], f1[u]);
                    }
                    uint4 d2[3];
                    uint32_t f2[3];
                    if (st + 2 < 5) {
#pragma unroll
                        for (int u = 0; u < 3; u++) ld_stage(ru[u], st + 2, d2[u], f2[u]);
                    }
                    const int kb = st < 4 ? 2 * st + (c8 >> 2) : 8;
                    // K-blocks 2st and 2st+1 are released by one commit pair
                    // after the same O^T MMAs: one wait covers both
                    const bool w = tc::mbar_wait(&kb_empty[st < 4 ? 2 * st : 8], (c & 1) ^ 1, a.err);
                    if (!__all_sync(0xffffffffu, w)) {  // the warp leaves together
                        ok = false;
                        break;
                    }
                    uint8_t *dst = rb + kb * kRBlock;
#pragma unroll
                    for (int u = 0; u < 3; u++) {
                        if (u >= nu) continue;
                        const int r = rw + 48 * u;
                        if (st < 4) {
                            const float scl = __uint_as_float(f0[u]);
                            range_bad |= kMaxE4M3 * fabsf(scl) > kMaxF16;
                            const __half s_hi = __float2half_rn(scl);
                            const __half2 shi2 = __half2half2(s_hi);
                            const __half2 slo2 = __half2half2(__float2half_rn(scl - __half2float(s_hi)));
                            const __nv_fp8x2_storage_t *pp = (const __nv_fp8x2_storage_t *)&d0[u];
                            uint32_t packed[8];
#pragma unroll
                            for (int e = 0; e < 8; e++) packed[e] = e4m3x2_scaled(pp[e], shi2, slo2);
                            const int q0 = (c8 & 3) * 2;
                            *(uint4 *)(dst + tc::sw128_offset(r, q0)) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                            *(uint4 *)(dst + tc::sw128_offset(r, q0 + 1)) = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                        } else {
                            range_bad |= bf16x8_beyond_f16(d0[u]);
                            *(uint4 *)(dst + tc::sw128_offset(r, c8r)) = bf16x8_to_f16x8(d0[u]);  // rope
                        }
                    }
                    tc::fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (st < 4) {
                            tc::mbar_arrive(&kb_full[2 * st]);
                            tc::mbar_arrive(&kb_full[2 * st + 1]);
                        } else {
                            tc::mbar_arrive(&kb_full[8]);
                        }
                    }
                    if (st == 4 && c8 == 0) {
                        // warm L2 with the next chunk's rows (their ids have
                        // arrived by now), so that its loads hit L2
#pragma unroll
                        for (int u = 0; u < 3; u++)
                            if (idn[u] >= 0 && idn[u] < a.max_row)
                                tc::prefetch_l2(a.pool + (size_t)unit_of(idn[u]) * 656, 656);
                    }
#pragma unroll
                    for (int u = 0; u < 3; u++) {
                        d0[u] = d1[u];
                        f0[u] = f1[u];
                        d1[u] = d2[u];
                        f1[u] = f2[u];
                    }
                }
            }
            // the softmax groups leave together when a wait ran out
            if (warp < 10 && !softmax_part(c, warp < 6 ? 0 : 32, std::true_type{})) {
                ok = false;
                break;
            }
            if (ok) issue_first();  // lands before PV(c) frees the first K-blocks
        }
        if (range_bad) set_error(a.err, HS_ERR_RANGE);
        if (a.cluster && warp < 10) {
            // ---- two splits in one cluster merge symmetrically over eight
            // warps (heads 0-31 on warps 2-5, 32-63 on warps 6-9; thread =
            // output dim row = TMEM lane): split s finishes output dims
            // [256 s, 256 s + 256) (O^T tiles 2s, 2s+1) and hands the peer its
            // other two tiles and its (max, sum) through distributed shared
            // memory.  Received layout in the row buffer: O as [tile 0..1]
            // [head/4][128 dims][4 heads] fp32 (consecutive threads on
            // consecutive 16 bytes), then max[64], sum[64]; the merged bf16
            // output is staged as [64 heads][256 dims] behind it and leaves in
            // 16-byte stores.
            const int sp = warp & 3;
            const int r = sp * 32 + lane;
            const uint32_t lane_base = tmem + ((uint32_t)(sp * 32) << 16);
            const int hb = warp < 6 ? 0 : 32;
            const bool fin = ok && nchunks > 0 && tc::mbar_wait(o_done, (nchunks - 1) & 1, a.err);
            const bool good = !bar_or_group(!fin);
            if (good) {
                tc::fence_after_sync();
                if (warp == 4) {  // every lane holds the same denominators
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        float lv[16];
                        tc::tmem_ld16(lane_base + l_col + 16 * q, lv);
                        tc::tmem_ld_wait();
                        if (lane == 0) {
#pragma unroll
                            for (int i = 0; i < 16; i++) lsum[16 * q + i] = lv[i];
                        }
                    }
                }
                bar_group();
            }
            const size_t g0 = (size_t)qr * a.H + hh * kTcHeads;  // first output head row
            const uint32_t peer = 1u - (uint32_t)split;
            float *rx = (float *)rb;
            float *rx_m = rx + 2 * 16 * 128 * 4;
            float *rx_l = rx_m + 64;
            __nv_bfloat16 *ostage = (__nv_bfloat16 *)(rb + 72 * 1024);
            // this CTA's row buffer is idle once every MMA completed
            // (relaxed: it hands over no data; this CTA's MMAs were seen done
            // through o_done above)
            if (warp == 4 && lane == 0) tc::mbar_arrive_remote_relaxed(tc::mapa(tc::smem_addr(peer_ready), peer));
            const bool w1 = tc::mbar_wait_cluster(peer_ready, 0, a.err);
            if (!bar_or_group(!w1)) {
                const uint32_t dst = tc::mapa(tc::smem_addr(rx), peer);
                for (int gi = 0; gi < 2; gi++) {
                    const int g = 2 * (int)peer + gi;
#pragma unroll
                    for (int h0 = hb; h0 < hb + 32; h0 += 16) {
                        float ov[16];
                        if (good) {
                            tc::tmem_ld16(lane_base + o_col + g * kTcHeads + h0, ov);
                            tc::tmem_ld_wait();
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; i++) ov[i] = 0.f;
                        }
#pragma unroll
                        for (int q4 = 0; q4 < 4; q4++) {
                            const int hq = (h0 >> 2) + q4;
                            const uint32_t at = dst + (uint32_t)((((gi * 16 + hq) * 128 + r) * 4) * 4);
                            tc::st_cluster_v4(at, ov[4 * q4], ov[4 * q4 + 1], ov[4 * q4 + 2], ov[4 * q4 + 3]);
                        }
                    }
                }
                if (warp < 6 && r < 64) {
                    const float l = good ? lsum[r] : 0.f;
                    tc::st_cluster_f32(tc::mapa(tc::smem_addr(rx_m + r), peer), l > 0.f ? mref[r] : -INFINITY);
                    tc::st_cluster_f32(tc::mapa(tc::smem_addr(rx_l + r), peer), l);
                }
            }
            // every thread's writes are ordered before its own arrival
            tc::mbar_arrive_remote(tc::mapa(tc::smem_addr(peer_data), peer));
            const bool w0 = tc::mbar_wait_cluster(peer_data, 0, a.err);
            if (!bar_or_group(!w0)) {
                float *wf = red;  // [0,64): own weight / L, [64,128): the peer's weight / L
                if (warp < 6 && r < 64) {
                    const float l0 = good ? lsum[r] : 0.f, l1 = rx_l[r];
                    const float m0 = l0 > 0.f ? mref[r] : -INFINITY, m1 = rx_m[r];
                    const float M = fmaxf(m0, m1);
                    const float w0v = m0 == -INFINITY ? 0.f : exp2f(m0 - M);
                    const float w1v = m1 == -INFINITY ? 0.f : exp2f(m1 - M);
                    const float Ls = l0 * w0v + l1 * w1v;
                    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
                    wf[r] = w0v * inv;
                    wf[64 + r] = w1v * inv;
                    if (a.lse && split == 0) a.lse[g0 + r] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
                }
                bar_group();
                for (int gi = 0; gi < 2; gi++) {
                    const int g = 2 * split + gi;
#pragma unroll
                    for (int h0 = hb; h0 < hb + 32; h0 += 16) {
                        float ov[16];
                        if (good) {
                            tc::tmem_ld16(lane_base + o_col + g * kTcHeads + h0, ov);
                            tc::tmem_ld_wait();
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; i++) ov[i] = 0.f;
                        }
#pragma unroll
                        for (int q4 = 0; q4 < 4; q4++) {
                            const int hq = (h0 >> 2) + q4;
                            const float4 pv = *(const float4 *)(rx + ((gi * 16 + hq) * 128 + r) * 4);
                            const float4 fa = *(const float4 *)(wf + 4 * hq);       // broadcast
                            const float4 fb = *(const float4 *)(wf + 64 + 4 * hq);  // broadcast
                            const float pp[4] = {pv.x, pv.y, pv.z, pv.w};
                            const float wa[4] = {fa.x, fa.y, fa.z, fa.w};
                            const float wb[4] = {fb.x, fb.y, fb.z, fb.w};
#pragma unroll
                            for (int e = 0; e < 4; e++) {
                                const int h = 4 * hq + e;
                                const float v = fmaf(ov[4 * q4 + e], wa[e], pp[e] * wb[e]);
                                ostage[h * 256 + gi * 128 + r] = __float2bfloat16(v);
                            }
                        }
                    }
                }
                bar_group();
                // 64 heads x 256 dims of bf16: 2048 16-byte vectors over 256 threads
                const int t = (warp - 2) * 32 + lane;
                for (int v = t; v < 64 * 32; v += 256) {
                    const int h = v >> 5, c16 = v & 31;
                    *(uint4 *)(a.out + (g0 + h) * kNope + split * 256 + c16 * 8) =
                        *(const uint4 *)(ostage + h * 256 + c16 * 8);
                }
            }
        } else if (!a.cluster && warp < 6) {  // epilogue: thread = output dim row = TMEM lane
            const int sp = warp & 3;
            const int r = sp * 32 + lane;
            const uint32_t lane_base = tmem + ((uint32_t)(sp * 32) << 16);
            // ---- epilogue
            const bool fin = ok && nchunks > 0 && tc::mbar_wait(o_done, (nchunks - 1) & 1, a.err);
            const bool good = !bar_or_softmax(!fin);
            if (good) {
                tc::fence_after_sync();
                // every lane holds the same denominators: stage them in smem
                if (sp == 0) {
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        float lv[16];
                        tc::tmem_ld16(lane_base + l_col + 16 * q, lv);
                        tc::tmem_ld_wait();
                        if (lane == 0) {
#pragma unroll
                            for (int i = 0; i < 16; i++) lsum[16 * q + i] = lv[i];
                        }
                    }
                }
                bar_softmax();
            }
            const size_t g0 = (size_t)qr * a.H + hh * kTcHeads;  // first output head row
            if (good) {
                for (int g = 0; g < 4; g++) {
                    const int d = g * 128 + r;
#pragma unroll
                    for (int h0 = 0; h0 < 64; h0 += 16) {
                        float ov[16];
                        tc::tmem_ld16(lane_base + o_col + g * kTcHeads + h0, ov);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; i++) {
                            const int h = h0 + i;
                            if (a.splits == 1) {
                                const float l = lsum[h];
                                a.out[(g0 + h) * kNope + d] = __float2bfloat16(l > 0.f ? ov[i] / l : 0.f);
                            } else {
                                a.part[((g0 + h) * a.splits + split) * (kNope + 2) + d] = ov[i];
                            }
                        }
                    }
                }
                if (r < 64) {
                    const float l = lsum[r], m = mref[r];
                    if (a.splits == 1) {
                        if (a.lse) a.lse[g0 + r] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
                    } else {
                        float *pp = a.part + ((g0 + r) * a.splits + split) * (kNope + 2);
                        pp[kNope] = l > 0.f ? m : -INFINITY;
                        pp[kNope + 1] = l;
                    }
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

size_t simt_smem() { return ((size_t)kHeadsPerCta * kLatent + (size_t)kChunk * kRowStride) * 4; }

}  // namespace

static int simt_splits(const hs_pool_config &c, int rows) {
    const int ctas = rows * (c.mla_heads / kHeadsPerCta);
    int s = (2 * kNumSMs + ctas - 1) / ctas;
    s = s < 1 ? 1 : (s > kMaxSplits ? kMaxSplits : s);
    const int maxs = (c.top_k + kChunk - 1) / kChunk;  // at least one chunk per split
    s = s > maxs ? maxs : s;
    const int kc = ((c.top_k + s - 1) / s + kChunk - 1) / kChunk * kChunk;
    return (c.top_k + kc - 1) / kc;
}

static bool tc_eligible(const hs_pool_config &c) {
    return c.row_fmt == HS_ROW_E4M3_656 && c.mla_heads % kTcHeads == 0;
}

// One CTA per SM (shared memory).  Cost in chunk times: waves x (chunks per
// CTA + about four chunks of start-up: query staging, TMEM allocation and
// the first chunk's load latency) + one for the combine pass when split.
static int tc_splits(const hs_pool_config &c, int rows) {
    const int chunks = (c.top_k + kTcRows - 1) / kTcRows;
    const int base = rows * (c.mla_heads / kTcHeads);
    int best = 1;
    long best_cost = -1;
    for (int s = 1; s <= chunks && s <= kMaxSplits; s++) {
        const long cps = (chunks + s - 1) / s;
        const long waves = ((long)base * s + kNumSMs - 1) / kNumSMs;
        const long cost = waves * (cps + 4) + (s > 1 ? 1 : 0);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    const int kc = ((c.top_k + best - 1) / best + kTcRows - 1) / kTcRows * kTcRows;
    return (c.top_k + kc - 1) / kc;
}

bool pair_eligible(const hs_pool *p);
int pair_splits(const hs_pool_config &c, int rows);
cudaError_t pair_setup(const hs_pool *p);
cudaError_t launch_pair_attention(const hs_pool *p, int layer, const void *q, const int32_t *row_id,
                                  int B, int nq, float scale, void *out, float *lse, cudaStream_t st,
                                  bool q_ready, bool pdl);

// Which tensor-core kernel a batch takes.  The pair kernel (the latent dims
// split over a 2-CTA cluster, every MMA at M = N = 128, each row converted
// once) wins when the batch fills the GPU with pairs: measured at 128 heads,
// K = 2048, 256 queries it takes 348 us per layer against 445 for the
// 64-head kernel; below about one wave of pairs its longer per-chunk chain
// (two exchanges between the CTAs per 128 rows) costs more than it saves (32
// queries: 70 against 62 us; 4 queries: 42 against 30 us).
constexpr int kPairMinQueryGroups = 64;  // queries x 128-head groups

static bool pair_cfg(const hs_pool_config &c, int rows) {
    return c.row_fmt == HS_ROW_E4M3_656 && c.mla_heads % 128 == 0 &&
           rows * (c.mla_heads / 128) >= kPairMinQueryGroups;
}

static int splits_for(const hs_pool_config &c, int rows) {
    if (pair_cfg(c, rows)) return pair_splits(c, rows);
    return tc_eligible(c) ? tc_splits(c, rows) : simt_splits(c, rows);
}

int attention_kernel_count(const hs_pool *p, int B, int nq) {
    const int s = splits_for(p->cfg, B * nq);
    if (pair_cfg(p->cfg, B * nq)) return s > 1 ? 2 : 1;
    if (tc_eligible(p->cfg)) return s > 2 ? 2 : 1;
    return s > 1 ? 2 : 1;
}

size_t attention_partial_floats(const hs_pool_config *c) {
    size_t worst = 0;
    const int nq = c->num_spec + 1;
    for (int rows = 1; rows <= c->max_requests * nq; rows++) {
        const int s = splits_for(*c, rows);
        if (s > 1) {
            const size_t need = (size_t)rows * c->mla_heads * s * (kNope + 2);
            worst = need > worst ? need : worst;
        }
    }
    return worst;
}

cudaError_t attention_setup(const hs_pool *p) {
    cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)simt_smem());
    if (e != cudaSuccess) return e;
    e = pair_setup(p);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                AttnTcSmem::bytes);
}

cudaError_t launch_attention(const hs_pool *p, int layer, const void *q, const int32_t *row_id,
                             int B, int nq, float scale, void *out, float *lse, cudaStream_t st,
                             bool q_ready, bool pdl) {
    const int rows = B * nq;
    const int K = p->cfg.top_k;
    const int splits = splits_for(p->cfg, rows);
    if (pair_cfg(p->cfg, rows) && pair_eligible(p)) {
        cudaError_t e = launch_pair_attention(p, layer, q, row_id, B, nq, scale, out, lse, st, q_ready, pdl);
        if (e != cudaSuccess) return e;
        if (splits > 1)
            attn_combine_kernel<<<rows * p->cfg.mla_heads, 128, 0, st>>>(p->d.attn_part, splits,
                                                                       (__nv_bfloat16 *)out, lse);
        return cudaGetLastError();
    }
    if (tc_eligible(p->cfg)) {
        AttnTcArgs a;
        a.q = (const __nv_bfloat16 *)q;
        a.row_id = row_id;
        a.pool = p->d.rows;
        a.layer = layer;
        a.L = p->cfg.num_mla_layers;
        a.P = p->cfg.page_tokens;
        a.H = p->cfg.mla_heads;
        a.K = K;
        a.splits = splits;
        a.kc = ((K + splits - 1) / splits + kTcRows - 1) / kTcRows * kTcRows;
        a.max_row = (int)(p->cfg.gpu_blocks * p->cfg.page_tokens);
        a.scale_log2 = scale * kLog2e;
        a.out = (__nv_bfloat16 *)out;
        a.lse = lse;
        a.part = p->d.attn_part;
        a.err = p->d.err;
        a.cluster = splits == 2;
        a.q_ready = q_ready;
        dim3 grid(rows, a.H / kTcHeads, splits);
        // the two splits of a (query, 64 heads) merge through DSMEM as a cluster
        PdlLaunch lc(grid, dim3(kAttnThreads), AttnTcSmem::bytes, st,
                     a.cluster ? dim3(1, 1, 2) : dim3(1, 1, 1), pdl);
        cudaError_t e = cudaLaunchKernelEx(&lc.cfg, attn_tc_kernel, a);
        if (e != cudaSuccess) return e;
    } else {
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
        a.K = K;
        a.splits = splits;
        a.kc = ((K + splits - 1) / splits + kChunk - 1) / kChunk * kChunk;
        a.scale_log2 = scale * kLog2e;
        a.out = (__nv_bfloat16 *)out;
        a.lse = lse;
        a.part = p->d.attn_part;
        a.max_row = (int)(p->cfg.gpu_blocks * p->cfg.page_tokens);
        a.err = p->d.err;
        dim3 grid(rows, a.H / kHeadsPerCta, splits);
        attn_simt_kernel<<<grid, 256, simt_smem(), st>>>(a);
    }
    if (splits > 2 || (splits == 2 && !tc_eligible(p->cfg)))  // 2 tensor-core splits merge in-cluster
        attn_combine_kernel<<<rows * p->cfg.mla_heads, 128, 0, st>>>(p->d.attn_part, splits,
                                                                   (__nv_bfloat16 *)out, lse);
    return cudaGetLastError();
}

cudaError_t indexer_setup(const hs_pool *p);
cudaError_t resolve_setup(const hs_pool *p);
cudaError_t topk_setup(const hs_pool *p);
cudaError_t dcp_setup(const hs_pool *p);

cudaError_t setup_kernel_attributes(const hs_pool *p) {
    cudaError_t e = indexer_setup(p);
    if (e == cudaSuccess) e = topk_setup(p);
    if (e == cudaSuccess) e = dcp_setup(p);
    if (e == cudaSuccess) e = resolve_setup(p);
    if (e == cudaSuccess) e = attention_setup(p);
    return e;
}

}  // namespace hs
