// Indexer score ("Un contexte d'un million sur huit H200", section "Ce qui se
// passe": the indexer scores every cached token; its cache stays resident).
//
//   s[b][j][t] = sum_h w[b][j][h] * ReLU(sigma[b][t] * (q[b][j][h][:] . k[b][t][:]))
//
// Tensor-core kernel (E4M3 keys, head dim 128, nq*Hi <= 256): the dense
// contraction D[token][(j,h)] = k[token] . q[j][h] runs on tcgen05 with FP8
// operands (kind::f8f6f4, fp32 accumulate):
//   A = 128 keys x 128 B (K-major, 128-byte swizzle), brought by TMA from the
//       request's key slab, kStages-deep ring;
//   B = the request's nq*Hi query rows (same layout), staged once per CTA;
//   D = 128 TMEM lanes x nq*Hi columns, two accumulators (double buffer).
// Warp 0 issues TMA, warp 1 issues MMAs, and G = min(nq, 4) groups of four
// epilogue warps (one thread per token = one TMEM lane) read D, apply ReLU,
// the head weights and sigma and write the scores (coalesced): group g takes
// queries g, g + G, ...  The epilogue is bound by instruction issue, so one
// warp per query and TMEM sub-partition gives each SMSP up to four warps to
// switch between while TMEM loads are in flight.  Every mbarrier wait is
// bounded.
//
// General kernel (any format / dims): one CTA per 128-token tile of one
// request; keys and queries decoded to fp32 in shared memory; each thread
// owns one token and loops over (query, head).
//
// All sums are fp32; with the synthetic inputs they are exact, so results
// do not depend on the order of summation (tensor core or not).
//
// The gate is ReLU (the lightning-indexer form).
#include <cuda_fp8.h>

#include "tc.cuh"

namespace hs {
namespace {

constexpr int kTile = 128;

__device__ __forceinline__ float gate(float x) { return x > 0.f ? x : 0.f; }

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
            acc = fmaf(wf[j * Hi + h], gate(x), acc);
        }
        scores[((size_t)b * nq + j) * stride + t] = acc;
    }
}


// ------------------------------------------------------------------------
// tensor-core path
// ------------------------------------------------------------------------
constexpr int kTcStages = 4;
constexpr int kTcMaxGroups = 4;  // epilogue warp groups (one per query)
constexpr int kTcThreads = 64 + 128 * kTcMaxGroups;
constexpr int kTileBytes = kTile * 128;  // 128 tokens x 128 B

struct IdxTcArgs {
    const uint8_t *q;  // [B][nq*Hi][128] E4M3
    const float *w;    // [B][nq*Hi]
    const float *ksc;  // [maxR][maxT]
    const int32_t *seq_len;
    float *scores;
    int64_t stride;
    int nq, Hi, maxT, tiles_per_cta, ncols, tmem_cols;
    int32_t *err;
};

// Shared memory of one CTA for ncols = nq * Hi query rows: the rows take
// ncols x 128 B (a multiple of 4 KB, since Hi % 32 == 0), so the key stages
// behind them stay 1024-aligned for the 128-byte swizzle.  Sizing the rows
// by ncols rather than the 256 maximum lets three CTAs share an SM at one
// query (three epilogue warps per TMEM sub-partition instead of two).
struct IdxTcSmem {
    __host__ __device__ static int k_off(int ncols) { return ncols * 128; }
    __host__ __device__ static int w_off(int ncols) { return k_off(ncols) + kTcStages * kTileBytes; }
    __host__ __device__ static int bar_off(int ncols) { return w_off(ncols) + 256 * 4; }
    __host__ __device__ static int tslot_off(int ncols) { return bar_off(ncols) + (2 * kTcStages + 5) * 8; }
    __host__ __device__ static int bytes(int ncols) { return tslot_off(ncols) + 16 + 1024; }  // + alignment slack
};

// sum_h w[h] * ReLU(d[h]) over nh columns of one TMEM lane row starting at
// taddr (nh a multiple of 32), in 32-column batches (both loads in flight,
// one wait) and eight independent partial sums.  fmaxf(d, 0) may give -0 for
// d = -0 where ReLU gives +0; the sums start at +0 and every product with a
// zero is a zero, so the total is the same.
template <int kNh>
__device__ __forceinline__ float weighted_relu_sum(uint32_t taddr, const float *wj, int nh) {
    float part[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const int n = kNh ? kNh : nh;
#pragma unroll
    for (int h0 = 0; h0 < (kNh ? kNh : 256); h0 += 32) {
        if (!kNh && h0 >= n) break;
        float v[32];
        tc::tmem_ld16(taddr + h0, v);
        tc::tmem_ld16(taddr + h0 + 16, v + 16);
        tc::tmem_ld_wait();
        const float4 *wq = (const float4 *)(wj + h0);
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const float4 wv = wq[u];  // shared-memory broadcast
            const int o = 4 * (u & 1);
            part[o] = fmaf(wv.x, fmaxf(v[4 * u], 0.f), part[o]);
            part[o + 1] = fmaf(wv.y, fmaxf(v[4 * u + 1], 0.f), part[o + 1]);
            part[o + 2] = fmaf(wv.z, fmaxf(v[4 * u + 2], 0.f), part[o + 2]);
            part[o + 3] = fmaf(wv.w, fmaxf(v[4 * u + 3], 0.f), part[o + 3]);
        }
    }
    return ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
}

// The waits of the producer and MMA threads.  Each try_wait may suspend the
// thread for up to kCtlSuspendNs and resumes it as soon as the phase
// completes, so a waiting control thread takes no issue slots from the
// epilogue warps that share its SM sub-partition (warps 0 and 1 sit on
// sub-partitions 0 and 1; with a plain retry loop there, a clock64 trace
// showed those epilogue warps about 15 % slower per tile than the others and
// the MMA of each tile waiting for them).  Bounded like tc::mbar_wait.
constexpr uint32_t kCtlSuspendNs = 1000000;  // at most 1 ms per look

__device__ __forceinline__ bool ctl_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P1;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2, %3;\n\t"
        "selp.b32 %0, 1, 0, P1;\n\t}"
        : "=r"(ok)
        : "r"(tc::smem_addr(bar)), "r"(parity), "r"(kCtlSuspendNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool ctl_wait(uint64_t *bar, uint32_t parity, int32_t *err) {
    if (ctl_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!ctl_try_wait(bar, parity)) {
        if (clock64() - t0 > tc::kWaitCycles) {
            set_error(err, HS_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Two fp32 lanes as one 64-bit operand of the packed f32x2 instructions.
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

// d = a * b + c in each of the two fp32 lanes (rounded like fmaf).
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ float2 unpack2(unsigned long long v) {
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
    return f;
}

// The 64-head sum of one query in 32-column batches (both loads of a batch
// in flight, one wait), the products through packed f32x2 FMAs (two heads
// per instruction) into eight partial sums.
__device__ __forceinline__ float weighted_relu_sum64(uint32_t taddr, const float *wj) {
    unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};  // +0 in every lane
#pragma unroll
    for (int h0 = 0; h0 < 64; h0 += 32) {
        float v[32];
        tc::tmem_ld16(taddr + h0, v);
        tc::tmem_ld16(taddr + h0 + 16, v + 16);
        tc::tmem_ld_wait();
        const float4 *wq = (const float4 *)(wj + h0);
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const float4 wv = wq[u];  // shared-memory broadcast
            const unsigned long long r0 = pack2(fmaxf(v[4 * u], 0.f), fmaxf(v[4 * u + 1], 0.f));
            const unsigned long long r1 = pack2(fmaxf(v[4 * u + 2], 0.f), fmaxf(v[4 * u + 3], 0.f));
            acc[(2 * u) & 3] = fma2(r0, pack2(wv.x, wv.y), acc[(2 * u) & 3]);
            acc[(2 * u + 1) & 3] = fma2(r1, pack2(wv.z, wv.w), acc[(2 * u + 1) & 3]);
        }
    }
    const float2 p0 = unpack2(acc[0]), p1 = unpack2(acc[1]), p2 = unpack2(acc[2]),
                 p3 = unpack2(acc[3]);
    return ((p0.x + p0.y) + (p1.x + p1.y)) + ((p2.x + p2.y) + (p3.x + p3.y));
}

__global__ void __launch_bounds__(kTcThreads, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap kmap, IdxTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *qs = smem;
    uint8_t *ks = smem + IdxTcSmem::k_off(a.ncols);
    float *wsm = (float *)(smem + IdxTcSmem::w_off(a.ncols));
    uint64_t *full = (uint64_t *)(smem + IdxTcSmem::bar_off(a.ncols));
    uint64_t *empty = full + kTcStages;
    uint64_t *tfull = empty + kTcStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *done = tempty + 2;
    uint32_t *tslot = (uint32_t *)(smem + IdxTcSmem::tslot_off(a.ncols));

    const int b = blockIdx.y;
    const int N = a.seq_len[b];
    const int ntiles = (N + kTile - 1) / kTile;
    const int tile0 = blockIdx.x * a.tiles_per_cta;
    const int tile1 = min(ntiles, tile0 + a.tiles_per_cta);
    if (tile0 >= tile1) return;  // uniform over the CTA
    const int nt = tile1 - tile0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // queries -> 128-byte-swizzled K-major rows; head weights -> smem
    const uint8_t *qb = a.q + (size_t)b * a.ncols * 128;
    for (int i = threadIdx.x; i < a.ncols * 8; i += blockDim.x) {
        const int r = i >> 3, c = i & 7;
        *(uint4 *)(qs + tc::sw128_offset(r, c)) = *(const uint4 *)(qb + r * 128 + c * 16);
    }
    for (int i = threadIdx.x; i < a.ncols; i += blockDim.x) wsm[i] = a.w[(size_t)b * a.ncols + i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; s++) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int k = 0; k < 2; k++) {
            tc::mbar_init(&tfull[k], 1);
            tc::mbar_init(&tempty[k], (int)blockDim.x - 64);  // every epilogue thread
        }
        tc::mbar_init(done, 1);
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tslot, a.tmem_cols);
        tc::tmem_relinquish();
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        if (lane == 0) {
            tc::prefetch_tensormap(&kmap);
            int issued = 0;
            for (int it = 0; it < nt; it++) {
                const int s = it % kTcStages;
                const uint32_t ph = (it / kTcStages) & 1;
                if (!ctl_wait(&empty[s], ph ^ 1, a.err)) break;
                tc::mbar_expect_tx(&full[s], kTileBytes);
                tc::tma_load_2d(ks + s * kTileBytes, &kmap, &full[s], 0,
                                b * a.maxT + (tile0 + it) * kTile);
                issued++;
            }
            // never leave with a copy in flight
            for (int it = max(0, issued - kTcStages); it < issued; it++)
                ctl_wait(&full[it % kTcStages], (it / kTcStages) & 1, a.err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tc::instr_desc(128, a.ncols, 0, 0, 0, 0);
            const uint32_t qaddr = tc::smem_addr(qs);
            for (int it = 0; it < nt; it++) {
                const int s = it % kTcStages;
                const uint32_t ph = (it / kTcStages) & 1;
                const int acc = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                if (!ctl_wait(&tempty[acc], aph ^ 1, a.err)) break;
                if (!ctl_wait(&full[s], ph, a.err)) break;
                tc::fence_after_sync();
                const uint32_t kaddr = tc::smem_addr(ks + s * kTileBytes);
#pragma unroll
                for (int kk = 0; kk < 4; kk++) {
                    const uint64_t ad = tc::smem_desc_sw128(kaddr + kk * 32, 16, 1024);
                    const uint64_t bd = tc::smem_desc_sw128(qaddr + kk * 32, 16, 1024);
                    tc::mma_f8f6f4(tmem + acc * a.ncols, ad, bd, idesc, kk > 0);
                }
                tc::mma_commit(&empty[s]);
                tc::mma_commit(&tfull[acc]);
            }
            // every MMA this thread issued has completed before TMEM is freed
            tc::mma_commit(done);
            ctl_wait(done, 0, a.err);
        }
    } else {
        const int sp = warp & 3;  // TMEM sub-partition this warp may read
        const int half = (warp - 2) >> 2;  // queries j = half, half + jstep, ...
        const int jstep = ((int)blockDim.x - 64) >> 7;  // the number of groups
        const int row = sp * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(sp * 32) << 16);
        const float *ksc = a.ksc + (size_t)b * a.maxT;
        int t = tile0 * kTile + row;
        float sig_next = t < N ? ksc[t] : 0.f;
        for (int it = 0; it < nt; it++) {
            const int acc = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            const float sig = sig_next;  // loaded one tile ahead
            if (it + 1 < nt && t + kTile < N) sig_next = ksc[t + kTile];
            const bool w = tc::mbar_wait(&tfull[acc], aph, a.err);
            if (!__all_sync(0xffffffffu, w)) break;  // the warp leaves together
            tc::fence_after_sync();
            const uint32_t tb = lane_base + acc * a.ncols;
            // per query (sigma > 0 comes out of the sum: sigma * ReLU(d) =
            // ReLU(sigma * d); with the power-of-two key scales of the
            // workloads both orders are exact)
            for (int j = half; j < a.nq; j += jstep) {
                const float accs = a.Hi == 64
                    ? weighted_relu_sum64(tb + j * a.Hi, wsm + j * a.Hi)
                    : weighted_relu_sum<0>(tb + j * a.Hi, wsm + j * a.Hi, a.Hi);
                if (t < N) a.scores[((size_t)b * a.nq + j) * a.stride + t] = sig * accs;
            }
            tc::fence_before_sync();
            tc::mbar_arrive(&tempty[acc]);
            t += kTile;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, a.tmem_cols);
    }
}

bool tc_eligible(const hs_pool *p, int nq) {
    const int ncols = nq * p->cfg.idx_heads;
    return p->cfg.idx_fmt == HS_IDX_E4M3 && p->cfg.idx_dim == 128 && p->cfg.idx_heads % 32 == 0 &&
           ncols >= 16 && ncols <= 256 && p->has_key_map;
}

int tmem_cols_for(int ncols) {
    int c = 32;
    while (c < 2 * ncols) c <<= 1;
    return c;
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
    e = cudaFuncSetAttribute(indexer_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             120 * 1024);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(indexer_simt_kernel<1>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
}

int indexer_kernel_count(const hs_pool *, int, int) { return 1; }

// Tiles per CTA for a grid of (chunks, B), given how many CTAs fit on one
// SM: minimise waves x (tiles per CTA + the fixed cost of starting a CTA,
// about four tiles' worth: TMEM allocation, query staging, pipeline fill).
static int pick_tiles_per_cta(int ntiles, int B, int per_sm) {
    const long slots = (long)kNumSMs * per_sm;
    int best = ntiles;
    double best_t = 1e30;
    for (int tpc = 1; tpc <= ntiles; tpc++) {
        const long chunks = (ntiles + tpc - 1) / tpc;
        const long ctas = chunks * B;
        const long waves = (ctas + slots - 1) / slots;
        const double t = (double)waves * (tpc + 4.0);
        if (t < best_t) {
            best_t = t;
            best = tpc;
        }
    }
    return best;
}

cudaError_t launch_indexer_score(const hs_pool *p, const void *q, const float *w, int B, int nq,
                                 float *scores, int64_t stride, cudaStream_t st) {
    const int maxT = p->cfg.max_tokens;
    if (tc_eligible(p, nq)) {
        IdxTcArgs a;
        a.q = (const uint8_t *)q;
        a.w = w;
        a.ksc = p->d.idx_scale;
        a.seq_len = p->d.seq_len;
        a.scores = scores;
        a.stride = stride;
        a.nq = nq;
        a.Hi = p->cfg.idx_heads;
        a.maxT = maxT;
        a.ncols = nq * p->cfg.idx_heads;
        a.tmem_cols = tmem_cols_for(a.ncols);
        a.err = p->d.err;
        const int per_sm_tmem = 512 / a.tmem_cols;
        const int per_sm_smem = (228 * 1024) / (IdxTcSmem::bytes(a.ncols) + 1024);
        const int per_sm = per_sm_tmem < per_sm_smem ? per_sm_tmem : per_sm_smem;
        // never co-schedule more CTAs than TMEM holds: pad the smem request
        int smem = IdxTcSmem::bytes(a.ncols);
        const int cap = (228 * 1024) / per_sm - 1024;
        if (per_sm == 1 && smem < 116 * 1024) smem = 116 * 1024;
        else if (smem < cap && per_sm_tmem < per_sm_smem) smem = cap;
        const int ntiles = (maxT + kTile - 1) / kTile;
        a.tiles_per_cta = pick_tiles_per_cta(ntiles, B, per_sm);
        dim3 grid((ntiles + a.tiles_per_cta - 1) / a.tiles_per_cta, B);
        // one group of four epilogue warps per query (up to four groups)
        const int threads = 64 + 128 * (nq < kTcMaxGroups ? nq : kTcMaxGroups);
        indexer_tc_kernel<<<grid, threads, smem, st>>>(p->key_map, a);
        return cudaGetLastError();
    }
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
