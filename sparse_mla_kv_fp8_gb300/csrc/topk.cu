// Top-K selection over indexer scores ("vLLM sert GLM-5.3 en contexte 1M sur
// 16 H200", section "Comment s'y prendre": the 2048 selected tokens).
//
// Radix select on an order-preserving 32-bit key of each fp32 score, 11 + 11
// + 10 bits, MSB first.  Each pass is one kernel over (chunk, row) CTAs that
// builds a shared-memory histogram of the still-undecided keys and adds it
// into a per-row global histogram with integer atomics (order independent);
// the last CTA of the row (ticket counter) picks the digit of the K-th
// largest key.  After three passes the threshold key T and the number `need`
// of keys equal to T to keep are known; two more kernels count, per chunk,
// keys above / equal to T and write the selected indices in ascending token
// order (keys equal to T are taken lowest index first).  Every count is an
// integer, so the result is bit-for-bit deterministic.
#include <algorithm>
#include <mutex>

#include "hs_internal.h"
#include "tc.cuh"

namespace hs {
namespace {

constexpr int kThreads = 1024;
constexpr int kPerThread = kTopkChunk / kThreads;

// Order-preserving key of an fp32 score.  -0 is first made +0: the two
// compare equal, so they must tie (and go to the lower token) like any other
// equal scores, not rank -0 below +0.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive scan over the block (blockDim.x a multiple of 32, <= 1024).
__device__ __forceinline__ int block_incl_scan(int v, int *warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int x = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += n;
        }
        warp_sums[lane] = x;
    }
    __syncthreads();
    if (warp > 0) v += warp_sums[warp - 1];
    __syncthreads();
    return v;
}

// vis is clamped to max_tokens: the later kernels read scores up to it, so a
// length beyond the score rows (a caller's device data) never reads past them.
__global__ void topk_init_kernel(TopkRowState *st, uint32_t *hist, const int32_t *seq_len,
                                 int nq, int K, int max_tokens) {
    const int row = blockIdx.x;
    const int b = row / nq, j = row - b * nq;
    const int vis = min(seq_len[b] - nq + j + 1, max_tokens);
    for (int i = threadIdx.x; i < kTopkBins; i += blockDim.x) hist[(size_t)row * kTopkBins + i] = 0;
    if (threadIdx.x == 0) {
        TopkRowState s;
        s.prefix = 0;
        s.mask = 0;
        s.need = K;
        s.take_all = vis <= K;
        s.ticket = 0;
        s.visible = vis > 0 ? vis : 0;
        s.pad[0] = s.pad[1] = 0;
        st[row] = s;
    }
}

__global__ void __launch_bounds__(kThreads) topk_hist_kernel(const float *__restrict__ scores,
                                                             int64_t stride, TopkRowState *st,
                                                             uint32_t *ghist, int pass) {
    __shared__ uint32_t sh[kTopkBins];
    __shared__ int warp_sums[32];
    __shared__ int is_last;
    const int row = blockIdx.y, chunk = blockIdx.x, tid = threadIdx.x;
    const TopkRowState s = st[row];
    if (s.take_all) return;  // uniform over the row's CTAs
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nbins = pass == 2 ? 1024 : 2048;
    for (int i = tid; i < nbins; i += kThreads) sh[i] = 0;
    __syncthreads();
    const int64_t base = (int64_t)chunk * kTopkChunk;
    const float *src = scores + (size_t)row * stride;
#pragma unroll
    for (int k = 0; k < kPerThread; k++) {
        const int64_t t = base + k * kThreads + tid;
        if (t < s.visible) {
            const uint32_t key = order_key(src[t]);
            if ((key & s.mask) == s.prefix) atomicAdd(&sh[(key >> shift) & (nbins - 1)], 1u);
        }
    }
    __syncthreads();
    uint32_t *gh = ghist + (size_t)row * kTopkBins;
    for (int i = tid; i < nbins; i += kThreads) {
        const uint32_t c = sh[i];
        if (c) atomicAdd(&gh[i], c);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = atomicAdd(&st[row].ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // Last CTA of this row: walk the bins from the largest key down.  Thread i
    // holds the two bins at descending positions 2i, 2i+1.
    int c0 = 0, c1 = 0;
    const int p0 = 2 * tid, p1 = 2 * tid + 1;
    if (p0 < nbins) c0 = (int)__ldcg(&gh[nbins - 1 - p0]);
    if (p1 < nbins) c1 = (int)__ldcg(&gh[nbins - 1 - p1]);
    const int incl = block_incl_scan(c0 + c1, warp_sums);
    const int above0 = incl - c0 - c1;  // keys in bins above position p0
    const int need = s.need;
    int found_pos = -1, found_above = 0;
    if (p0 < nbins && above0 < need && need <= above0 + c0) {
        found_pos = p0;
        found_above = above0;
    } else if (p1 < nbins && above0 + c0 < need && need <= above0 + c0 + c1) {
        found_pos = p1;
        found_above = above0 + c0;
    }
    if (found_pos >= 0) {
        const uint32_t bin = (uint32_t)(nbins - 1 - found_pos);
        TopkRowState n = s;
        n.prefix = s.prefix | (bin << shift);
        n.mask = s.mask | ((uint32_t)(nbins - 1) << shift);
        n.need = need - found_above;
        n.ticket = 0;
        st[row] = n;
    }
    // clear the row histogram for the next pass
    for (int i = tid; i < kTopkBins; i += kThreads) gh[i] = 0;
}

__global__ void __launch_bounds__(kThreads) topk_count_kernel(const float *__restrict__ scores,
                                                              int64_t stride,
                                                              const TopkRowState *st,
                                                              int32_t *chunk_cnt, int nchunks) {
    __shared__ int warp_sums[32];
    const int row = blockIdx.y, chunk = blockIdx.x, tid = threadIdx.x;
    const TopkRowState s = st[row];
    const int64_t base = (int64_t)chunk * kTopkChunk;
    const float *src = scores + (size_t)row * stride;
    int gt = 0, eq = 0;
#pragma unroll
    for (int k = 0; k < kPerThread; k++) {
        const int64_t t = base + k * kThreads + tid;
        if (t < s.visible) {
            if (s.take_all) {
                gt++;
            } else {
                const uint32_t key = order_key(src[t]);
                gt += key > s.prefix;
                eq += key == s.prefix;
            }
        }
    }
    const int packed = block_incl_scan((eq << 16) | gt, warp_sums);
    if (tid == kThreads - 1) {
        int32_t *c = chunk_cnt + ((size_t)row * nchunks + chunk) * 2;
        c[0] = packed & 0xFFFF;
        c[1] = packed >> 16;
    }
}

__global__ void __launch_bounds__(kThreads) topk_write_kernel(const float *__restrict__ scores,
                                                              int64_t stride,
                                                              const TopkRowState *st,
                                                              const int32_t *chunk_cnt,
                                                              int nchunks, int K, int32_t *topk) {
    __shared__ int warp_sums[32];
    __shared__ int before[2], total[2];
    const int row = blockIdx.y, chunk = blockIdx.x, tid = threadIdx.x;
    const TopkRowState s = st[row];
    const int need = s.take_all ? 0 : s.need;
    if (tid < 32) {
        int bg = 0, be = 0, tg = 0, te = 0;
        for (int c = tid; c < nchunks; c += 32) {
            const int g = chunk_cnt[((size_t)row * nchunks + c) * 2];
            const int e = chunk_cnt[((size_t)row * nchunks + c) * 2 + 1];
            tg += g;
            te += e;
            if (c < chunk) {
                bg += g;
                be += e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            bg += __shfl_xor_sync(0xffffffffu, bg, o);
            be += __shfl_xor_sync(0xffffffffu, be, o);
            tg += __shfl_xor_sync(0xffffffffu, tg, o);
            te += __shfl_xor_sync(0xffffffffu, te, o);
        }
        if (tid == 0) {
            before[0] = bg;
            before[1] = be;
            total[0] = tg;
            total[1] = te;
        }
    }
    __syncthreads();
    const int64_t base = (int64_t)chunk * kTopkChunk + (int64_t)tid * kPerThread;
    const float *src = scores + (size_t)row * stride;
    uint8_t flag[kPerThread];  // 1 = above T, 2 = equal to T
    int gt = 0, eq = 0;
#pragma unroll
    for (int k = 0; k < kPerThread; k++) {
        const int64_t t = base + k;
        flag[k] = 0;
        if (t < s.visible) {
            if (s.take_all) {
                flag[k] = 1;
            } else {
                const uint32_t key = order_key(src[t]);
                flag[k] = key > s.prefix ? 1 : (key == s.prefix ? 2 : 0);
            }
            gt += flag[k] == 1;
            eq += flag[k] == 2;
        }
    }
    const int v = (eq << 16) | gt;
    const int excl = block_incl_scan(v, warp_sums) - v;
    int gb = before[0] + (excl & 0xFFFF);
    int eb = before[1] + (excl >> 16);
    int32_t *out = topk + (size_t)row * K;
#pragma unroll
    for (int k = 0; k < kPerThread; k++) {
        if (flag[k] == 1) {
            out[gb + min(eb, need)] = (int32_t)(base + k);
            gb++;
        } else if (flag[k] == 2) {
            if (eb < need) out[gb + eb] = (int32_t)(base + k);
            eb++;
        }
    }
    if (chunk == 0) {
        const int taken = total[0] + min(total[1], need);
        for (int i = taken + tid; i < K; i += kThreads) out[i] = -1;
    }
}

// ---------------------------------------------------------------------------
// One-launch top-K for rows of up to 8 x 1024 x 32 tokens.  A row is owned by
// a cluster of G CTAs (1024 threads each); thread t of CTA g holds the keys of
// tokens g*1024*E + t*E + [0, E) in registers, so the scores are read once.
// The same three radix passes run on those registers: each CTA builds its
// shared-memory histogram, the cluster barrier publishes it, and every CTA
// sums the G histograms over distributed shared memory and takes the same
// decision.  Selected indices are then written in ascending order from
// block scans plus the totals of the lower-ranked CTAs.  All counts are
// integers: the result equals the multi-kernel path's bit for bit.
// ---------------------------------------------------------------------------
constexpr int kClusterThreads = 1024;
constexpr int kClusterMax = 8;
constexpr int kClusterSmem = (8 + 2) * kTopkBins * 4;  // histogram copies + merged pair

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

constexpr int kHistCopies = 8;  // per-warp-group histograms: fewer colliding atomics

template <int E>
__global__ void __launch_bounds__(kClusterThreads, 1)
topk_cluster_kernel(const float *__restrict__ scores, int64_t stride, int vec4,
                    const int32_t *seq_len, int nq, int K, int32_t *topk) {
    extern __shared__ __align__(16) uint32_t tk_smem[];
    uint32_t *copies = tk_smem;                            // [kHistCopies][2048]
    uint32_t *merged = tk_smem + kHistCopies * kTopkBins;  // [2][2048], read by the cluster
    __shared__ int warp_sums[32];
    __shared__ uint32_t decided[3];  // prefix, mask, need of the next pass
    __shared__ int totals[2];        // this CTA's keys above / equal to T
    const int G = gridDim.x, g = (int)cta_rank(), row = blockIdx.y, tid = threadIdx.x;
    // the histogram copies start zeroed (each merge below re-zeroes them);
    // this shared-memory setup may overlap the previous kernel's tail
    for (int i = tid; i < kHistCopies * kTopkBins / 4; i += kClusterThreads)
        ((uint4 *)copies)[i] = make_uint4(0, 0, 0, 0);
    tc::grid_dep_launch();
    tc::grid_dep_wait();
    const int b = row / nq, j = row - b * nq;
    const int vis = max(0, seq_len[b] - nq + j + 1);
    const bool take_all = vis <= K;
    const int64_t base = ((int64_t)g * kClusterThreads + tid) * E;
    const float *src = scores + (size_t)row * stride;

    uint32_t key[E];
    uint32_t valid = 0;  // bit e: token base + e is visible
#pragma unroll
    for (int e = 0; e < E; e += 4) {
        const int64_t t = base + e;
        if (vec4 && t + 3 < vis) {
            const float4 f = *(const float4 *)(src + t);
            key[e] = order_key(f.x);
            key[e + 1] = order_key(f.y);
            key[e + 2] = order_key(f.z);
            key[e + 3] = order_key(f.w);
            valid |= 0xFu << e;
        } else {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                key[e + i] = 0;
                if (t + i < vis) {
                    key[e + i] = order_key(src[t + i]);
                    valid |= 1u << (e + i);
                }
            }
        }
    }

    uint32_t prefix = 0, mask = 0, need = take_all ? 0u : (uint32_t)K;
    if (!take_all) {  // uniform over the cluster: every CTA of the row sees vis
        uint32_t *mine = copies + (threadIdx.x >> 5) % kHistCopies * kTopkBins;
#pragma unroll 1
        for (int pass = 0; pass < 3; pass++) {
            const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
            const int nbins = pass == 2 ? 1024 : 2048;
            __syncthreads();
#pragma unroll
            for (int e = 0; e < E; e++) {
                if (((valid >> e) & 1u) && (key[e] & mask) == prefix)
                    atomicAdd(&mine[(key[e] >> shift) & (uint32_t)(nbins - 1)], 1u);
            }
            __syncthreads();
            // this CTA's histogram: the copies summed
            uint32_t *h = merged + (pass & 1) * kTopkBins;
            for (int i = tid; i < nbins; i += kClusterThreads) {
                uint32_t c = 0;
#pragma unroll
                for (int k = 0; k < kHistCopies; k++) {
                    c += copies[k * kTopkBins + i];
                    copies[k * kTopkBins + i] = 0;  // ready for the next pass
                }
                h[i] = c;
            }
            // every CTA's histogram is complete and visible to the cluster
            tc::cluster_sync();
            // thread t: descending positions 4t .. 4t+3 (bins nbins-1-4t ...),
            // summed over the cluster with one 16-byte load per CTA
            uint32_t c4[4] = {0u, 0u, 0u, 0u};
            const bool mine4 = 4 * tid < nbins;
            if (mine4) {
                const uint32_t at = tc::smem_addr(&h[nbins - 4 - 4 * tid]);
                uint4 v[kClusterMax];
#pragma unroll
                for (int r = 0; r < kClusterMax; r++)
                    v[r] = r < G ? ld_cluster_v4(tc::mapa(at, (uint32_t)r)) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int r = 0; r < kClusterMax; r++) {
                    c4[0] += v[r].w;  // descending: bin nbins-1-4t first
                    c4[1] += v[r].z;
                    c4[2] += v[r].y;
                    c4[3] += v[r].x;
                }
            }
            const int sum4 = (int)(c4[0] + c4[1] + c4[2] + c4[3]);
            const int incl = block_incl_scan(sum4, warp_sums);
            int above = incl - sum4;
            const int nd = (int)need;
            if (mine4) {
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    if (above < nd && nd <= above + (int)c4[q]) {
                        const uint32_t bin = (uint32_t)(nbins - 1 - (4 * tid + q));
                        decided[0] = prefix | (bin << shift);
                        decided[1] = mask | ((uint32_t)(nbins - 1) << shift);
                        decided[2] = (uint32_t)(nd - above);
                    }
                    above += (int)c4[q];
                }
            }
            __syncthreads();
            prefix = decided[0];
            mask = decided[1];
            need = decided[2];
            // (the next pass writes the other merged buffer; this one is
            // rewritten two passes later, after every CTA has passed the
            // next cluster barrier and so finished reading it)
        }
    }

    // keys above / equal to the threshold T = prefix, in token order
    int gt = 0, eq = 0;
#pragma unroll
    for (int e = 0; e < E; e++) {
        if ((valid >> e) & 1u) {
            gt += take_all || key[e] > prefix;
            eq += !take_all && key[e] == prefix;
        }
    }
    const int v = (eq << 16) | gt;  // at most 1024 * 32 of each
    const int incl = block_incl_scan(v, warp_sums);
    if (tid == kClusterThreads - 1) {
        totals[0] = incl & 0xFFFF;
        totals[1] = incl >> 16;
    }
    tc::cluster_sync();
    int bg = 0, be = 0, tg = 0, te = 0;
    uint32_t tv[2 * kClusterMax];
#pragma unroll
    for (int r = 0; r < kClusterMax; r++) {
        tv[2 * r] = r < G ? ld_cluster_u32(tc::mapa(tc::smem_addr(&totals[0]), (uint32_t)r)) : 0u;
        tv[2 * r + 1] = r < G ? ld_cluster_u32(tc::mapa(tc::smem_addr(&totals[1]), (uint32_t)r)) : 0u;
    }
#pragma unroll
    for (int r = 0; r < kClusterMax; r++) {
        tg += (int)tv[2 * r];
        te += (int)tv[2 * r + 1];
        if (r < g) {
            bg += (int)tv[2 * r];
            be += (int)tv[2 * r + 1];
        }
    }
    const int excl = incl - v;
    bg += excl & 0xFFFF;
    be += excl >> 16;
    int32_t *out = topk + (size_t)row * K;
    const int nd = (int)need;
#pragma unroll
    for (int e = 0; e < E; e++) {
        if (!((valid >> e) & 1u)) continue;
        if (take_all || key[e] > prefix) {
            out[bg + min(be, nd)] = (int32_t)(base + e);
            bg++;
        } else if (key[e] == prefix) {
            if (be < nd) out[bg + be] = (int32_t)(base + e);
            be++;
        }
    }
    if (g == 0) {
        const int taken = tg + min(te, nd);
        for (int i = taken + tid; i < K; i += kClusterThreads) out[i] = -1;
    }
    tc::cluster_sync();  // peers may still be reading this CTA's totals
}

// ---------------------------------------------------------------------------
// Sampled-threshold top-K (K <= kTopkSampledMaxK, rows of any length).
//
// The radix passes above touch every score three times, with an atomic per
// still-undecided key, and at K / N of a few percent almost every key is
// decided against the threshold long before the last digit.  This path
// touches each score once, with a compare:
//   1. topk_thresh_kernel, one CTA per row: T = the order key of the r-th
//      largest of S scores of the row (S / 8 runs of 8 consecutive tokens
//      at evenly spaced positions), with r chosen so that about
//      m = max(2.5 K, 2048) tokens are expected at or above T (a sample
//      quantile: relative spread about 1 / sqrt(r), r >= 80 here).  Rows of
//      at most kTopkCandCap visible tokens take T = 0: all are candidates.
//   2. topk_filter_kernel, persistent warps over 512-token tiles: one
//      coalesced pass; every visible token with key >= T is appended (key,
//      token) to the row's candidate list, one atomic per warp and tile
//      reserving its range.
//   3. topk_select_kernel, per row one CTA or a cluster of one CTA per
//      131,072-token window.  When the row kept between K and kTopkCandCap
//      candidates, they contain every token of the exact top-K: the K-th
//      largest key of the row is then >= T, and every token at or above T
//      is a candidate.  An exact selection over the candidates (held in
//      registers; 12-bit digits of key - min) gives the threshold key and
//      the number of keys equal to it to take; bitmaps over the windows then
//      place the selection in ascending token order, equal keys lowest token
//      first.  When the sample misjudged the row (fewer than K or more than
//      the cap), one CTA runs the exact selection over the whole row instead.
// Either way the result is the multi-kernel path's, bit for bit.
// ---------------------------------------------------------------------------
// Tokens the sampled threshold aims to keep per row: 2.5 K, at least 2048.
// With the sample sizes below (r >= 80 of the sampled scores at or above
// the threshold) the kept count stays within +-60 % of this, so between K
// and the 8192-candidate cap, by more than five times its spread.
__host__ __device__ constexpr int64_t sampled_target(int K) {
    return (5 * (int64_t)K) / 2 > 2048 ? (5 * (int64_t)K) / 2 : 2048;
}

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelE = kTopkCandCap / kSelThreads;  // candidates per thread
constexpr int kFiltThreads = 256;
constexpr int kFiltE = 16;                         // scores per lane and tile
constexpr int kFiltTile = 32 * kFiltE;             // tokens per warp tile
constexpr int kDigitBins = 4096;                   // 12-bit digits
constexpr int kCoarseBins = kDigitBins / 32;
constexpr int kWinWords = 4096;                    // bitmap words per window
constexpr int kWinTokens = kWinWords * 32;
constexpr int kWordsPer = kWinWords / kSelThreads;  // 16, consecutive per thread
// Thread t's words sit at t * 17 + q: the 32 lanes reading their q-th words
// hit 32 different banks.
constexpr int kWinPadded = kWinWords / kWordsPer * (kWordsPer + 1);
__device__ __forceinline__ int padded_word(int w) { return w + w / kWordsPer; }

// Shared memory of a selecting CTA: the digit histograms while the
// threshold is found, then the window bitmaps.  16-byte aligned: the
// histograms are cleared and read with 16-byte accesses.
struct __align__(16) SelSmem {
    union {
        struct {
            uint32_t fine[kDigitBins];     // keys in play per digit
            uint32_t coarse[kCoarseBins];  // per 32 consecutive digits
        } h;
        struct {
            uint32_t gt[kWinPadded], eq[kWinPadded];
        } w;
    };
    uint32_t decided[3];
    int warp_sums[32];
    int tot[2];
    uint32_t few[32];  // the keys of a digit small enough for one warp
    int nfew;
};
// The select kernel's dynamic shared memory: SelSmem, the packed counts of
// the selected tokens before each bitmap word, the candidates' tokens, then
// the selection in output order (copied out coalesced).
constexpr size_t kSelPreOff = sizeof(SelSmem);
constexpr size_t kSelTokOff = kSelPreOff + (size_t)kWinPadded * 4;
constexpr size_t kSelOutOff = kSelTokOff + (size_t)kTopkCandCap * 4;
constexpr size_t kSelDynSmem = kSelOutOff + (size_t)kTopkSampledMaxK * 4;

__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Block-wide smallest and largest of the keys, returned to every thread.
__device__ __forceinline__ void block_minmax(uint32_t &lo, uint32_t &hi, SelSmem &sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) {
        sm.h.coarse[warp] = lo;
        sm.h.coarse[32 + warp] = hi;
    }
    __syncthreads();
    if (warp == 0) {
        uint32_t a = lane < kSelWarps ? sm.h.coarse[lane] : 0xFFFFFFFFu;
        uint32_t b = lane < kSelWarps ? sm.h.coarse[32 + lane] : 0u;
        a = __reduce_min_sync(0xffffffffu, a);
        b = __reduce_max_sync(0xffffffffu, b);
        if (lane == 0) {
            sm.decided[0] = a;
            sm.decided[1] = b;
        }
    }
    __syncthreads();
    lo = sm.decided[0];
    hi = sm.decided[1];
}

// Digit selection over the key range [lo, hi] of the keys still in play.
// The digit of a key is (key - lo) >> shift, with shift chosen so that the
// range spans at most 4096 digits: unlike the key's own high bits, these
// split the range the keys occupy evenly, also where it straddles a power
// of two (keys 0x3FF... and 0x400... share no high bits).  The digit that
// holds the need-th largest key narrows the range for the next pass; a
// pass with shift 0 ends on the exact key.
struct DigitRange {
    uint32_t lo, hi;
    int shift;  // of the next pass; -1 once lo is the key
    __device__ __forceinline__ void start(uint32_t l, uint32_t h) {
        lo = l;
        hi = h;
        shift = lo == hi ? -1 : max(0, 32 - __clz(hi - lo) - 12);
    }
    __device__ __forceinline__ bool in(uint32_t k) const { return k >= lo && k <= hi; }
    __device__ __forceinline__ uint32_t digit(uint32_t k) const { return (k - lo) >> shift; }
};

__device__ __forceinline__ void zero_hist(SelSmem &sm) {
    uint4 *h = (uint4 *)sm.h.fine;  // fine and coarse are contiguous
    for (int i = threadIdx.x; i < (kDigitBins + kCoarseBins) / 4; i += kSelThreads)
        h[i] = make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void count_key(SelSmem &sm, const DigitRange &r, uint32_t k) {
    const uint32_t d = r.digit(k);
    atomicAdd(&sm.h.fine[d], 1u);
    atomicAdd(&sm.h.coarse[d >> 5], 1u);
}

// After a counting pass: warp 0 finds the digit holding the need-th largest
// key, first among the coarse bins (lane l holds coarse bins 127 - 4l - q,
// top down), then among the 32 digits of that coarse bin; every thread then
// narrows its range to the digit and takes the rank within it.
__device__ __forceinline__ void digit_decide(SelSmem &sm, DigitRange &r, uint32_t &need) {
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        const int nd = (int)need;
        const uint4 c4 = *(const uint4 *)(sm.h.coarse + kCoarseBins - 4 - 4 * lane);
        const int cs[4] = {(int)c4.w, (int)c4.z, (int)c4.y, (int)c4.x};
        const int sum = cs[0] + cs[1] + cs[2] + cs[3];
        const int incl = warp_incl_scan(sum);
        const int above = incl - sum;
        const int src = __ffs(__ballot_sync(0xffffffffu, above < nd && nd <= incl)) - 1;
        int C = 0, base = 0, a = above;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            if (a < nd && nd <= a + cs[q]) {
                C = kCoarseBins - 1 - 4 * lane - q;
                base = a;
            }
            a += cs[q];
        }
        C = __shfl_sync(0xffffffffu, C, src);
        base = __shfl_sync(0xffffffffu, base, src);
        const int f = (int)sm.h.fine[32 * C + 31 - lane];
        const int fa = base + warp_incl_scan(f) - f;
        if (fa < nd && nd <= fa + f) {  // exactly one lane
            sm.decided[0] = (uint32_t)(32 * C + 31 - lane);
            sm.decided[1] = (uint32_t)(nd - fa);
            sm.decided[2] = (uint32_t)f;
        }
    }
    __syncthreads();
    const uint32_t d = sm.decided[0];
    need = sm.decided[1];
    const uint32_t lo = r.lo + (d << r.shift);
    const unsigned long long top = (unsigned long long)lo + ((1ull << r.shift) - 1ull);
    r.start(lo, top < r.hi ? (uint32_t)top : r.hi);
}

// Exact selection over keys held in registers: key e of thread t is the
// (e * 256 + t)-th of n.  Returns the key of the need-th largest (1 <= need
// <= n) and leaves in `need` how many keys equal to it are among the need
// largest.
template <int E>
__device__ uint32_t block_select(const uint32_t (&key)[E], int n, uint32_t &need, SelSmem &sm) {
    const int tid = threadIdx.x;
    uint32_t lo = 0xFFFFFFFFu, hi = 0;
#pragma unroll
    for (int e = 0; e < E; e++) {
        if (e * kSelThreads + tid < n) {
            lo = min(lo, key[e]);
            hi = max(hi, key[e]);
        }
    }
    block_minmax(lo, hi, sm);
    DigitRange r;
    r.start(lo, hi);
#pragma unroll 1
    while (r.shift >= 0) {  // uniform over the CTA
        __syncthreads();  // the previous reads of the histograms are done
        zero_hist(sm);
        if (tid == 0) sm.nfew = 0;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; e++)
            if (e * kSelThreads + tid < n && r.in(key[e])) count_key(sm, r, key[e]);
        __syncthreads();
        digit_decide(sm, r, need);
        if (r.shift >= 0 && sm.decided[2] <= 32u) {
            // at most 32 keys left in the range: gather them and let one
            // warp rank them against each other
            const int cnt = (int)sm.decided[2];
#pragma unroll
            for (int e = 0; e < E; e++)
                if (e * kSelThreads + tid < n && r.in(key[e])) sm.few[atomicAdd(&sm.nfew, 1)] = key[e];
            __syncthreads();
            if (tid < 32) {
                const uint32_t k = tid < cnt ? sm.few[tid] : 0u;
                int gt = 0, eq = 0;
                for (int j = 0; j < cnt; j++) {
                    const uint32_t o = sm.few[j];
                    gt += o > k;
                    eq += o == k;
                }
                if (tid < cnt && gt < (int)need && (int)need <= gt + eq) {  // same values
                    sm.decided[0] = k;
                    sm.decided[1] = need - (uint32_t)gt;
                }
            }
            __syncthreads();
            need = sm.decided[1];
            return sm.decided[0];
        }
    }
    return r.lo;
}

// Write this thread's share of a selection in ascending token order.  gt /
// eq hold the thread's tokens above / equal to the threshold as bits of
// consecutive tokens t0 + [0, 32); g and eb count the tokens above / equal
// before them; equal keys are taken while fewer than `need` came before.
__device__ __forceinline__ void emit_ordered(uint32_t gt, uint32_t eq, int64_t t0, int &g, int &eb,
                                             int need, int32_t *out) {
    uint32_t bits = gt | eq;
    while (bits) {
        const int i = __ffs(bits) - 1;
        bits &= bits - 1;
        const int32_t t = (int32_t)(t0 + i);
        if ((gt >> i) & 1u) {
            out[g + min(eb, need)] = t;
            g++;
        } else {
            if (eb < need) out[g + eb] = t;
            eb++;
        }
    }
}

// Sampled threshold of one row: the key of the r-th largest of S = E * 256
// scores, taken as S / 8 runs of 8 consecutive tokens centred at
// ((2j + 1) * vis) / (2 * S / 8), j < S / 8.
template <int E>
__global__ void __launch_bounds__(kSelThreads) topk_thresh_kernel(const float *__restrict__ scores,
                                                                  int64_t stride,
                                                                  const int32_t *seq_len, int nq,
                                                                  int K, int max_tokens,
                                                                  TopkRowState *st) {
    __shared__ SelSmem sm;
    const int row = blockIdx.x, tid = threadIdx.x;
    tc::grid_dep_launch();
    tc::grid_dep_wait();
    const int b = row / nq, j = row - b * nq;
    const int vis = max(0, min(seq_len[b] - nq + j + 1, max_tokens));
    const bool take_all = vis <= K;
    uint32_t T = 0;
    if (!take_all && vis > kTopkCandCap) {  // uniform over the CTA
        constexpr int S = E * kSelThreads;
        const int64_t m = sampled_target(K);
        const int r = (int)max((int64_t)1, min((int64_t)S, ((int64_t)S * m + vis - 1) / vis));
        const float *src = scores + (size_t)row * stride;
        // S / 8 runs of 8 consecutive scores (one 32-byte sector each),
        // centred at evenly spaced tokens; consecutive threads read a run
        constexpr int kRuns = S / 8;
        uint32_t key[E];
#pragma unroll
        for (int e = 0; e < E; e++) {
            const int i = e * kSelThreads + tid, run = i >> 3;
            const int64_t c = ((2 * (int64_t)run + 1) * vis) / (2 * kRuns);
            const int64_t first = min(max(c - 4, (int64_t)0), (int64_t)vis - 8);  // vis > 8192
            key[e] = order_key(src[first + (i & 7)]);
        }
        uint32_t need = (uint32_t)r;
        T = block_select<E>(key, S, need, sm);
    }
    if (tid == 0) {
        TopkRowState s;
        s.prefix = T;
        s.mask = 0;
        s.need = K;
        s.take_all = take_all;
        s.ticket = 0;  // candidates appended so far
        s.visible = vis;
        s.pad[0] = s.pad[1] = 0;
        st[row] = s;
    }
}

// Persistent filter: every warp walks tiles of 512 tokens (16 per lane) with
// a stride of the grid's warp count, tiles of consecutive rows side by side
// (so the warps in flight spread their atomics over the rows' counters), and
// holds the next tile's scores in registers while it handles the current
// one, so its loads stay in flight across the candidate atomic.  Scores are
// read up to the row capacity (inside every score row), masked to the
// visible tokens only in the tile that holds the end of the row.  V4: rows
// are 16-byte aligned, a lane reads float4s.
template <bool V4>
__global__ void __launch_bounds__(kFiltThreads, 4) topk_filter_kernel(const float *__restrict__ scores,
                                                                      int64_t stride, int max_tokens,
                                                                      int rows, TopkRowState *st,
                                                                      uint2 *cand) {
    const int lane = threadIdx.x & 31;
    const int tiles = (max_tokens + kFiltTile - 1) / kFiltTile;
    const uint32_t wstride = gridDim.x * (kFiltThreads / 32);
    tc::grid_dep_launch();
    tc::grid_dep_wait();
    // element e of this lane is token base + tok_off(e): lane-interleaved
    // float4s (V4) or lane-interleaved scores
    auto tok_off = [&](int e) -> int { return V4 ? 4 * (32 * (e >> 2) + lane) + (e & 3) : 32 * e + lane; };
    auto load = [&](int row, int tile, float (&v)[kFiltE]) {
        const int base = tile * kFiltTile;
        const float *src = scores + (size_t)row * stride + base;
        const int lim = max_tokens - base;  // tokens of this tile inside the row capacity
        if (V4) {
#pragma unroll
            for (int k = 0; k < kFiltE / 4; k++) {
                const int o = tok_off(4 * k);
                float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
                if (o + 3 < lim) {
                    f = __ldcs((const float4 *)(src + o));
                } else {
                    if (o < lim) f.x = src[o];
                    if (o + 1 < lim) f.y = src[o + 1];
                    if (o + 2 < lim) f.z = src[o + 2];
                }
                v[4 * k] = f.x;
                v[4 * k + 1] = f.y;
                v[4 * k + 2] = f.z;
                v[4 * k + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < kFiltE; e++) {
                const int o = tok_off(e);
                v[e] = o < lim ? src[o] : 0.f;
            }
        }
    };
    auto handle = [&](int row, int tile, const float (&v)[kFiltE]) {
        const int base = tile * kFiltTile;
        const int vis = __ldg(&st[row].visible);
        if (__ldg(&st[row].take_all) || base >= vis) return;  // uniform over the warp
        const uint32_t T = __ldg(&st[row].prefix);
        uint32_t hit = 0;
        if (base + kFiltTile <= vis) {
#pragma unroll
            for (int e = 0; e < kFiltE; e++) hit |= (uint32_t)(order_key(v[e]) >= T) << e;
        } else {
#pragma unroll
            for (int e = 0; e < kFiltE; e++)
                hit |= (uint32_t)(base + tok_off(e) < vis && order_key(v[e]) >= T) << e;
        }
        if (!__any_sync(0xffffffffu, hit)) return;
        const int c = __popc(hit);
        const int incl = warp_incl_scan(c);
        uint32_t pos = 0;
        if (lane == 31) pos = atomicAdd(&st[row].ticket, (uint32_t)incl);
        pos = __shfl_sync(0xffffffffu, pos, 31) + (uint32_t)(incl - c);
        uint2 *dst = cand + (size_t)row * kTopkCandCap;
#pragma unroll
        for (int e = 0; e < kFiltE; e++) {  // entries past the cap are counted, not stored
            if ((hit >> e) & 1u) {
                if (pos < (uint32_t)kTopkCandCap)
                    dst[pos] = make_uint2(order_key(v[e]), (uint32_t)(base + tok_off(e)));
                pos++;
            }
        }
    };
    // tile id = tile * rows + row; the warp's ids advance by wstride, so
    // (row, tile) advance by (wstride % rows, wstride / rows) with a carry
    const uint32_t w0 = blockIdx.x * (kFiltThreads / 32) + (threadIdx.x >> 5);
    const int drow = (int)(wstride % (uint32_t)rows), dtile = (int)(wstride / (uint32_t)rows);
    int row = (int)(w0 % (uint32_t)rows), tile = (int)(w0 / (uint32_t)rows);
    auto advance = [&](int &r, int &t) {
        r += drow;
        t += dtile;
        if (r >= rows) {
            r -= rows;
            t++;
        }
    };
    float a[kFiltE], b[kFiltE];  // two tiles in turn: one in flight, one handled
    if (tile < tiles) load(row, tile, a);
#pragma unroll 1
    while (tile < tiles) {
        int nrow = row, ntile = tile;
        advance(nrow, ntile);
        if (ntile < tiles) load(nrow, ntile, b);
        handle(row, tile, a);
        row = nrow;
        tile = ntile;
        if (tile >= tiles) break;
        advance(nrow, ntile);
        if (ntile < tiles) load(nrow, ntile, a);
        handle(row, tile, b);
        row = nrow;
        tile = ntile;
    }
}

// The exact selection over a whole row from its scores (the select kernel's
// path for rows whose sampled threshold kept too few or too many tokens).
__device__ void select_whole_row(const float *__restrict__ src, int vis, int K, int32_t *out,
                                 SelSmem &sm) {
    const int tid = threadIdx.x;
    uint32_t lo = 0xFFFFFFFFu, hi = 0, need = (uint32_t)K;
    for (int t = tid; t < vis; t += kSelThreads) {
        const uint32_t key = order_key(src[t]);
        lo = min(lo, key);
        hi = max(hi, key);
    }
    block_minmax(lo, hi, sm);
    DigitRange r;
    r.start(lo, hi);
#pragma unroll 1
    while (r.shift >= 0) {  // uniform over the CTA
        __syncthreads();
        zero_hist(sm);
        __syncthreads();
        for (int t = tid; t < vis; t += kSelThreads) {
            const uint32_t key = order_key(src[t]);
            if (r.in(key)) count_key(sm, r, key);
        }
        __syncthreads();
        digit_decide(sm, r, need);
    }
    const uint32_t T = r.lo;
    // ordered write, in tiles of 256 x 32 tokens (32 consecutive per thread)
    int g0 = 0, e0 = 0;
#pragma unroll 1
    for (int64_t tile = 0; tile < vis; tile += 32 * kSelThreads) {
        const int64_t t0 = tile + 32 * (int64_t)tid;
        uint32_t gt = 0, eq = 0;
#pragma unroll 4
        for (int i = 0; i < 32; i++) {
            if (t0 + i < vis) {
                const uint32_t key = order_key(src[t0 + i]);
                gt |= (uint32_t)(key > T) << i;
                eq |= (uint32_t)(key == T) << i;
            }
        }
        const int v = (__popc(eq) << 16) | __popc(gt);  // at most 8192 of each per tile
        const int incl = block_incl_scan(v, sm.warp_sums);
        if (tid == kSelThreads - 1) {
            sm.tot[0] = incl & 0xFFFF;
            sm.tot[1] = incl >> 16;
        }
        const int excl = incl - v;
        int g = g0 + (excl & 0xFFFF), eb = e0 + (excl >> 16);
        emit_ordered(gt, eq, t0, g, eb, (int)need, out);
        __syncthreads();
        g0 += sm.tot[0];
        e0 += sm.tot[1];
    }
}

// One CTA per row and token window: with G = gridDim.x > 1 the row's G CTAs
// form a cluster, CTA g marks and places window g, and each CTA learns how
// many selected tokens the windows before its own hold from their CTAs'
// totals over distributed shared memory; with G = 1 one CTA walks the
// windows in turn.  Each CTA finds the threshold itself from the row's
// candidates (the same result in every CTA).
__global__ void __launch_bounds__(kSelThreads, 2)
topk_select_kernel(const float *__restrict__ scores, int64_t stride, const TopkRowState *st,
                   const uint2 *cand, int K, int32_t *topk) {
    extern __shared__ __align__(16) uint8_t sel_dyn[];
    SelSmem &sm = *(SelSmem *)sel_dyn;
    uint32_t *pre = (uint32_t *)(sel_dyn + kSelPreOff);  // [kWinPadded]
    uint32_t *toks = (uint32_t *)(sel_dyn + kSelTokOff);  // [kTopkCandCap]
    int32_t *obuf = (int32_t *)(sel_dyn + kSelOutOff);    // [K]
    const int G = gridDim.x, g = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
    tc::grid_dep_launch();
    tc::grid_dep_wait();
    const TopkRowState s = st[row];
    const int vis = s.visible;
    int32_t *out = topk + (size_t)row * K;
    if (s.take_all) {  // (the row's CTAs all take this path or none)
        if (g == 0)
            for (int i = tid; i < K; i += kSelThreads) out[i] = i < vis ? i : -1;
        return;
    }
    const uint32_t n = s.ticket;
    if (n < (uint32_t)K || n > (uint32_t)kTopkCandCap) {  // uniform over the row's CTAs
        if (g == 0) select_whole_row(scores + (size_t)row * stride, vis, K, out, sm);
        return;
    }
    const uint2 *src = cand + (size_t)row * kTopkCandCap;
    uint32_t key[kSelE];
#pragma unroll
    for (int e = 0; e < kSelE; e++) {
        const uint32_t i = (uint32_t)(e * kSelThreads + tid);
        const uint2 v = i < n ? __ldcg(src + i) : make_uint2(0u, 0u);
        key[e] = v.x;
        toks[i] = v.y;
    }
    uint32_t need = (uint32_t)K;
    const uint32_t T = block_select<kSelE>(key, (int)n, need, sm);
    const int nd = (int)need;

    // One window [w0, w0 + kWinTokens): mark the candidates at or above T in
    // two bitmaps, count the marks before every word (block scan over
    // threads holding 16 consecutive words each) into pre[] and the window's
    // totals into sm.tot.
    auto count_window = [&](int w0) -> uint32_t {
        __syncthreads();  // the histograms / the previous window are read
        for (int i = tid; i < 2 * kWinPadded; i += kSelThreads)
            sm.w.gt[i] = 0;  // gt and eq are contiguous
        __syncthreads();
        uint32_t mine = 0;  // bit e: candidate e of this thread is marked in this window
#pragma unroll
        for (int e = 0; e < kSelE; e++) {
            const int i = e * kSelThreads + tid;
            const int off = (int)toks[i] - w0;
            if (i < (int)n && key[e] >= T && off >= 0 && off < kWinTokens) {
                atomicOr((key[e] > T ? sm.w.gt : sm.w.eq) + padded_word(off >> 5), 1u << (off & 31));
                mine |= 1u << e;
            }
        }
        __syncthreads();
        int v = 0;  // packed (equal << 16) | above of this thread's words
#pragma unroll
        for (int q = 0; q < kWordsPer; q++) {
            const int pw = tid * (kWordsPer + 1) + q;
            v += (__popc(sm.w.eq[pw]) << 16) | __popc(sm.w.gt[pw]);
        }
        const int incl = block_incl_scan(v, sm.warp_sums);  // at most kTopkCandCap of each
        if (tid == kSelThreads - 1) {
            sm.tot[0] = incl & 0xFFFF;
            sm.tot[1] = incl >> 16;
        }
        int run = incl - v;
#pragma unroll
        for (int q = 0; q < kWordsPer; q++) {
            const int pw = tid * (kWordsPer + 1) + q;
            pre[pw] = (uint32_t)run;
            run += (__popc(sm.w.eq[pw]) << 16) | __popc(sm.w.gt[pw]);
        }
        __syncthreads();
        return mine;
    };
    // Every marked candidate of the window takes its output position from
    // those counts, with g0 / e0 tokens above / equal to T in the windows
    // before; it is written to obuf[position - pbase].
    auto place_window = [&](int w0, uint32_t mine, int g0, int e0, int pbase) {
#pragma unroll
        for (int e = 0; e < kSelE; e++) {
            if ((mine >> e) & 1u) {
                const int i = e * kSelThreads + tid, off = (int)toks[i] - w0;
                const int pw = padded_word(off >> 5);
                const uint32_t below = (1u << (off & 31)) - 1u, pk = pre[pw];
                const int gb = g0 + (int)(pk & 0xFFFFu) + __popc(sm.w.gt[pw] & below);
                const int eb = e0 + (int)(pk >> 16) + __popc(sm.w.eq[pw] & below);
                if (key[e] > T) obuf[gb + min(eb, nd) - pbase] = (int32_t)toks[i];
                else if (eb < nd) obuf[gb + eb - pbase] = (int32_t)toks[i];
            }
        }
    };
    if (G == 1) {
        int g0 = 0, e0 = 0;
#pragma unroll 1
        for (int w0 = 0; w0 < vis; w0 += kWinTokens) {
            const uint32_t mine = count_window(w0);
            place_window(w0, mine, g0, e0, 0);
            g0 += sm.tot[0];
            e0 += sm.tot[1];
        }
        __syncthreads();
        for (int i = tid; i < K; i += kSelThreads) out[i] = obuf[i];  // exactly K were written
        return;
    }
    // cluster: window g only (G covers the row capacity, so a window past
    // vis simply holds nothing)
    const int w0 = g * kWinTokens;
    const uint32_t mine = count_window(w0);
    tc::cluster_sync();  // every CTA's totals are in its shared memory
    int g0 = 0, e0 = 0;
    for (int r = 0; r < g; r++) {
        g0 += (int)ld_cluster_u32(tc::mapa(tc::smem_addr(&sm.tot[0]), (uint32_t)r));
        e0 += (int)ld_cluster_u32(tc::mapa(tc::smem_addr(&sm.tot[1]), (uint32_t)r));
    }
    // the window's selected tokens fill output positions [p0, p1)
    const int p0 = g0 + min(e0, nd), p1 = g0 + sm.tot[0] + min(e0 + sm.tot[1], nd);
    place_window(w0, mine, g0, e0, p0);
    __syncthreads();
    for (int i = tid; i < p1 - p0; i += kSelThreads) out[p0 + i] = obuf[i];
    tc::cluster_sync();  // the peers have read this CTA's totals
}

// Elements per thread for the one-launch path, or 0 when rows are too long.
// Measured on GB300 with rows of 65,536 tokens: 16 keys per thread (4-CTA
// clusters) beat 8 keys (8-CTA clusters: 38.9 against 21.6 us at 16 rows)
// and 32 keys (2-CTA clusters: 28.7 against 22.5 us at 32 rows): the cluster
// barriers and distributed-shared-memory merges grow with the cluster, the
// histogram work with the keys per thread.  So 16 keys per thread while
// every row's CTAs fit one wave; otherwise 32, whose rows cost fewer CTA-
// microseconds (2 x 28.7 against 4 x 22.5) and fit one wave up to twice as
// many rows.
int cluster_elems(int max_tokens, int rows) {
    auto ctas = [&](int e) { return (max_tokens + kClusterThreads * e - 1) / (kClusterThreads * e); };
    if (ctas(16) <= kClusterMax && (int64_t)rows * ctas(16) <= kNumSMs) return 16;
    return ctas(32) <= kClusterMax ? 32 : 0;
}

}  // namespace

cudaError_t topk_setup(const hs_pool *) {
    cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kClusterSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(topk_cluster_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kClusterSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSelDynSmem);
    return e;
}

// The sampled-threshold path, unless every row's cluster of the one-launch
// kernel fits one wave with 16 keys per thread: there that kernel's single
// launch measured faster (22.5 against about 30 us at 32 rows of 65,536).
bool use_sampled(const hs_pool *p, int rows) {
    return p->d.topk_cand && cluster_elems(p->cfg.max_tokens, rows) != 16;
}

int topk_kernel_count(const hs_pool *p, int B, int nq) {
    if (use_sampled(p, B * nq)) return 3;
    return cluster_elems(p->cfg.max_tokens, B * nq) ? 1 : 6;
}

cudaError_t launch_topk(const hs_pool *p, const float *scores, int64_t stride, int B, int nq,
                        int32_t *topk, cudaStream_t st) {
    const int rows = B * nq, nch = p->topk_nchunks, K = p->cfg.top_k;
    const int vec4 = ((uintptr_t)scores % 16 == 0) && (stride % 4 == 0);
    if (use_sampled(p, rows)) {  // K <= kTopkSampledMaxK
        const int maxT = p->cfg.max_tokens;
        // 4096 samples while they put r >= 128 at the longest row, else 16384
        const int64_t m = sampled_target(K);
        const bool wide = 128 * (int64_t)maxT > 4096 * m;
        PdlLaunch lt(dim3((unsigned)rows), dim3(kSelThreads), 0, st);
        cudaError_t e = wide ? cudaLaunchKernelEx(&lt.cfg, topk_thresh_kernel<64>, scores, stride,
                                                  (const int32_t *)p->d.seq_len, nq, K, maxT,
                                                  p->d.topk_state)
                             : cudaLaunchKernelEx(&lt.cfg, topk_thresh_kernel<16>, scores, stride,
                                                  (const int32_t *)p->d.seq_len, nq, K, maxT,
                                                  p->d.topk_state);
        if (e != cudaSuccess) return e;
        const int64_t warps = (int64_t)rows * ((maxT + kFiltTile - 1) / kFiltTile);
        const int fgrid = (int)std::min<int64_t>((warps + 7) / 8, 4 * kNumSMs);
        PdlLaunch lf(dim3((unsigned)fgrid), dim3(kFiltThreads), 0, st);
        e = vec4 ? cudaLaunchKernelEx(&lf.cfg, topk_filter_kernel<true>, scores, stride, maxT, rows,
                                      p->d.topk_state, p->d.topk_cand)
                 : cudaLaunchKernelEx(&lf.cfg, topk_filter_kernel<false>, scores, stride, maxT, rows,
                                      p->d.topk_state, p->d.topk_cand);
        if (e != cudaSuccess) return e;
        // one CTA per row and token window (a cluster) while the windows of
        // the row capacity number 2-8 and every row's CTAs fit one wave (two
        // per SM), else one CTA walking them: each CTA repeats the
        // threshold search, so a second wave costs more than the windows
        // save (measured at 4 rows of 2^20 tokens: 69 -> 48 us for the
        // top-K; at 256 rows of 142,000: 84 -> 100 us)
        const int windows = (maxT + kWinTokens - 1) / kWinTokens;
        const int Gw = windows >= 2 && windows <= 8 && (int64_t)rows * windows <= 2 * kNumSMs ? windows : 1;
        PdlLaunch ls(dim3((unsigned)Gw, (unsigned)rows), dim3(kSelThreads), kSelDynSmem, st,
                     dim3((unsigned)Gw, 1, 1));
        return cudaLaunchKernelEx(&ls.cfg, topk_select_kernel, scores, stride,
                                  (const TopkRowState *)p->d.topk_state,
                                  (const uint2 *)p->d.topk_cand, K, topk);
    }
    const int E = cluster_elems(p->cfg.max_tokens, rows);
    if (E) {
        const int G = (p->cfg.max_tokens + kClusterThreads * E - 1) / (kClusterThreads * E);
        PdlLaunch lc(dim3((unsigned)G, (unsigned)rows), dim3(kClusterThreads), kClusterSmem, st,
                     dim3((unsigned)G, 1, 1));
        if (E == 16)
            return cudaLaunchKernelEx(&lc.cfg, topk_cluster_kernel<16>, scores, stride, vec4,
                                      (const int32_t *)p->d.seq_len, nq, K, topk);
        return cudaLaunchKernelEx(&lc.cfg, topk_cluster_kernel<32>, scores, stride, vec4,
                                  (const int32_t *)p->d.seq_len, nq, K, topk);
    }
    topk_init_kernel<<<rows, 256, 0, st>>>(p->d.topk_state, p->d.topk_hist, p->d.seq_len, nq, K,
                                            p->cfg.max_tokens);
    dim3 grid(nch, rows);
    for (int pass = 0; pass < 3; pass++)
        topk_hist_kernel<<<grid, kThreads, 0, st>>>(scores, stride, p->d.topk_state,
                                                    p->d.topk_hist, pass);
    topk_count_kernel<<<grid, kThreads, 0, st>>>(scores, stride, p->d.topk_state,
                                                 p->d.topk_chunk, nch);
    topk_write_kernel<<<grid, kThreads, 0, st>>>(scores, stride, p->d.topk_state,
                                                 p->d.topk_chunk, nch, K, topk);
    return cudaGetLastError();
}

}  // namespace hs

// ---------------------------------------------------------------------------
// Top-K without any allocation.
//
// Some callers cannot allocate device memory at all: a serving engine that
// reserved most of the GPU for its own block pool at start-up (so a later
// cudaMalloc fails or fragments that pool), or host code that must not make
// the device-wide synchronising allocation calls.  For them the radix top-K
// also runs on a scratch area that lives in this library's own static device
// memory, with no pool and no workspace argument.  Every GPU that loads the
// library holds that area (kNoAllocScratchBytes) until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxRows = 64;                      // B * nq
constexpr int kNoAllocMaxTokens = 1 << 20;               // tokens per request
constexpr int kNoAllocMaxChunks = kNoAllocMaxTokens / hs::kTopkChunk;
constexpr size_t kNoAllocStateBytes = sizeof(hs::TopkRowState) * kNoAllocMaxRows;
constexpr size_t kNoAllocHistBytes = sizeof(uint32_t) * hs::kTopkBins * kNoAllocMaxRows;
constexpr size_t kNoAllocChunkBytes = sizeof(int32_t) * 2 * kNoAllocMaxChunks * kNoAllocMaxRows;
constexpr size_t kNoAllocScratchBytes = kNoAllocStateBytes + kNoAllocHistBytes + kNoAllocChunkBytes;
static_assert(kNoAllocStateBytes % 256 == 0 && kNoAllocHistBytes % 256 == 0, "scratch carving");

// The scratch itself.  Host code must never pass this name to a kernel: on
// the host it only stands for the symbol.  Its device address comes from
// cudaGetSymbolAddress, taken once per device below.
static __device__ __align__(256) uint8_t g_topk_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
uint8_t *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (set up on first use).
cudaError_t noalloc_scratch(uint8_t **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_topk_noalloc_scratch);
        if (e != cudaSuccess || !p) return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
        g_noalloc_ptr[dev] = (uint8_t *)p;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" hs_status hs_topk_noalloc(const float *scores, int64_t score_stride,
                                     const int32_t *seq_len, int32_t B, int32_t nq, int32_t K,
                                     int32_t max_tokens, int32_t *topk, cudaStream_t stream) {
    if (!scores || !seq_len || !topk || B <= 0 || nq <= 0 || K <= 0 || max_tokens <= 0 ||
        score_stride < max_tokens)
        return HS_ERR_INVALID_ARG;
    if ((int64_t)B * nq > kNoAllocMaxRows || max_tokens > kNoAllocMaxTokens)
        return HS_ERR_CAPACITY;  // beyond the static scratch
    uint8_t *base = nullptr;
    if (noalloc_scratch(&base) != cudaSuccess) {
        cudaGetLastError();
        return HS_ERR_CUDA;
    }
    hs::TopkRowState *state = (hs::TopkRowState *)base;
    uint32_t *hist = (uint32_t *)(base + kNoAllocStateBytes);
    int32_t *chunk = (int32_t *)(base + kNoAllocStateBytes + kNoAllocHistBytes);
    const int rows = B * nq;
    const int nch = (max_tokens + hs::kTopkChunk - 1) / hs::kTopkChunk;
    // the init kernel clears the histograms and the per-row state that the
    // previous call left behind (the chunk counts are fully rewritten), and
    // clamps each row's visible length to max_tokens, so a seq_len[b] beyond
    // it reads no score past the caller's rows
    hs::topk_init_kernel<<<rows, 256, 0, stream>>>(state, hist, seq_len, nq, K, max_tokens);
    dim3 grid(nch, rows);
    for (int pass = 0; pass < 3; pass++)
        hs::topk_hist_kernel<<<grid, hs::kThreads, 0, stream>>>(scores, score_stride, state, hist,
                                                                pass);
    hs::topk_count_kernel<<<grid, hs::kThreads, 0, stream>>>(scores, score_stride, state, chunk,
                                                             nch);
    hs::topk_write_kernel<<<grid, hs::kThreads, 0, stream>>>(scores, score_stride, state, chunk,
                                                             nch, K, topk);
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}
