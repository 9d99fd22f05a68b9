// Fused top-K resolve ("Un contexte d'un million sur huit H200", section "Les
// trois états de résidence"): a selected token whose page is on the GPU is
// read in place; a token already in the request's hot buffer refreshes its
// LRU entry; a miss copies exactly one row per layer from pinned host memory
// into a hot-buffer slot.  No CPU decision: the step counter, the victim
// choice and the copy list all live on the device.
//
// resolve_plan_kernel: one 1024-thread CTA per request.
//   1. validate the nq lists (ascending, -1 padded, inside the request);
//   2. merge them into U, their sorted union without duplicates (the set
//      bits of a bitmap over the request's tokens, whose per-word counts also
//      index U in step 6; beyond 262,144 tokens merge-path ranks by binary
//      search, then a compaction of first occurrences);
//   3. classify each u in U: resident page -> in place; hot_map[u] >= 0 -> hit
//      (stamp = step); else miss; misses are compacted in ascending order;
//   4. choose victims: among slots with stamp < step, the M smallest keys
//      (stamp, slot), found by an 8-bit-digit radix select on the stamp plus a
//      lowest-slot-first cut among equal stamps; victims are compacted in
//      ascending slot order (fewer such slots than misses: every one of them
//      is a victim, the misses beyond read nothing, HS_ERR_CAPACITY);
//   5. the i-th miss takes the i-th victim: hot_map / slot_token / stamp are
//      updated and the (token, slot) pair goes to the device miss list;
//   6. every (j, k) entry gets its pool row id (with one list, U is the list
//      and each entry's row id is written as soon as its slot is known).
// miss_copy_kernel: a grid-stride copy of the miss list, 16-byte vectors,
// consecutive threads on consecutive bytes of a row (coalesced on both the
// host-link read and the HBM write).
#include "hs_internal.h"
#include "tc.cuh"

namespace hs {
namespace {

constexpr int kThreads = 1024;

__device__ __forceinline__ int block_excl_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += n;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int y = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += n;
        }
        warp_sums[lane] = y;
    }
    __syncthreads();
    const int incl = x + (warp > 0 ? warp_sums[warp - 1] : 0);
    *total = warp_sums[nw - 1];
    __syncthreads();
    return incl - v;
}

// Stable compaction of indices [0, n) for which pred holds; emit(i, rank).
template <class Pred, class Emit>
__device__ __forceinline__ int block_compact(int n, Pred pred, Emit emit, int *warp_sums) {
    const int seg = (n + kThreads - 1) / kThreads;
    const int lo = min(n, (int)threadIdx.x * seg), hi = min(n, lo + seg);
    int c = 0;
    for (int i = lo; i < hi; i++) c += pred(i) ? 1 : 0;
    int total;
    int r = block_excl_scan(c, warp_sums, &total);
    for (int i = lo; i < hi; i++)
        if (pred(i)) emit(i, r++);
    __syncthreads();
    return total;
}

__device__ __forceinline__ int lower_bound(const int32_t *a, int n, int32_t x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < x) lo = mid + 1; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ int upper_bound(const int32_t *a, int n, int32_t x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= x) lo = mid + 1; else hi = mid;
    }
    return lo;
}

struct PlanArgs {
    const int32_t *topk;
    int nq, K, P, C, hot_pages, maxT, max_pages, L, R;
    const int32_t *seq_len;
    const int32_t *block_table;
    int32_t *hot_map;
    int32_t *slot_token;
    uint32_t *stamp;
    const int32_t *hot_blocks;
    uint32_t *req_step;
    int32_t *miss_count;
    int32_t *miss_tok;
    int32_t *miss_slot;
    int32_t *row_id;
    int32_t *err;
    unsigned long long *stats;
    int words;  // > 0: union of several lists by a bitmap of this many words over the tokens
    int stage_pages;  // > 0: the request's block table is staged in shared memory
};

__global__ void __launch_bounds__(kThreads, 1) resolve_plan_kernel(PlanArgs a) {
    extern __shared__ int32_t sm[];
    __shared__ int warp_sums[32];
    __shared__ int lens[8];
    __shared__ uint32_t hist[256];
    __shared__ int sel[4];
    const int b = blockIdx.x, tid = threadIdx.x;
    tc::grid_dep_launch();
    const int n = a.nq * a.K;
    int32_t *lst = sm;            // [n] the lists; later: index into U of each miss
    int32_t *merged = lst + n;    // [n] merged lists; later: miss tokens
    int32_t *U = merged + n;      // [n] sorted unique union
    int32_t *uslot = U + n;       // [n] -1 resident, >= 0 slot, -2 miss, -3 unserved
    int32_t *victim = uslot + n;  // [n] victim slots, ascending
    // The request's length and block table change only through copies from
    // the host, ordered on the stream before every kernel of the step: the
    // table's used pages are staged while the previous kernel still runs
    // (behind the bitmap and its word counts, [stage_pages]).
    const int N = a.seq_len[b];
    const int32_t *bt = a.block_table + (size_t)b * a.max_pages;
    if (a.stage_pages > 0) {
        int32_t *bts = victim + n + 2 * a.words;
        const int np = min(a.stage_pages, (N + a.P - 1) / a.P);
        for (int i = tid; i < np; i += kThreads) bts[i] = bt[i];
        bt = bts;  // read after the __syncthreads below
    }
    tc::grid_dep_wait();  // the lists (and the previous plan's step count) come from earlier kernels
    const uint32_t step = a.req_step[b] + 1;
    const int32_t *tk = a.topk + (size_t)b * n;
    int32_t *rid = a.row_id + (size_t)b * n;
    const size_t hm = (size_t)b * a.maxT, sc = (size_t)b * a.C;
    const int32_t *hb = a.hot_blocks + (size_t)b * a.hot_pages;

    // 1. load and validate
    if (tid < 8) lens[tid] = 0;
    for (int i = tid; i < n; i += kThreads) lst[i] = tk[i];
    __syncthreads();
    bool bad = false;
    for (int i = tid; i < n; i += kThreads) {
        const int k = i % a.K;
        const int32_t v = lst[i];
        if (v < -1 || v >= N) bad = true;
        if (k + 1 < a.K) {
            const int32_t w = lst[i + 1];
            if (v == -1 ? (w != -1) : (w != -1 && w <= v)) bad = true;
        }
        if (v >= 0 && (k + 1 == a.K || lst[i + 1] == -1)) lens[i / a.K] = k + 1;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) {
            set_error(a.err, HS_ERR_INDEX_RANGE);
            a.miss_count[b] = 0;
        }
        for (int i = tid; i < n; i += kThreads) rid[i] = -1;
        return;
    }

    // 2. merge-path ranks -> merged (ties: lower list first), then dedup into
    // U.  One list is its own union (validated ascending, no duplicates).
    const bool single = a.nq == 1;
    int nu;
    int32_t *miss, *missidx;  // scratch for step 4, whichever arrays are dead by then
    if (single) {
        nu = lens[0];
        miss = merged;
        missidx = U;
        U = lst;
    } else if (a.words > 0) {
        // Each list is ascending without repeats (validated above), so the
        // union is the set bits of a bitmap over the request's tokens, in
        // order; each word's count of the bits before it then gives a
        // token's index in U without a search (step 6).  Thread t owns
        // words [t * wpt, (t + 1) * wpt).
        uint32_t *bm = (uint32_t *)(victim + n);
        int32_t *wpre = (int32_t *)(bm + a.words);
        const int words = (N + 31) >> 5;  // N <= max_tokens: words <= a.words
        for (int w = tid; w < words; w += kThreads) bm[w] = 0u;
        __syncthreads();
        for (int i = tid; i < n; i += kThreads) {
            const int32_t x = lst[i];
            if (x >= 0) atomicOr(&bm[x >> 5], 1u << (x & 31));
        }
        __syncthreads();
        const int wpt = (words + kThreads - 1) / kThreads;
        const int w0 = min(words, tid * wpt), w1 = min(words, w0 + wpt);
        int cnt = 0;
        for (int w = w0; w < w1; w++) cnt += __popc(bm[w]);
        int run = block_excl_scan(cnt, warp_sums, &nu);
        for (int w = w0; w < w1; w++) {
            wpre[w] = run;
            uint32_t bits = bm[w];
            while (bits) {
                U[run++] = (w << 5) + __ffs(bits) - 1;
                bits &= bits - 1;
            }
        }
        __syncthreads();
        miss = merged;  // merged is unused on this path
        missidx = lst;  // lists are dead now
    } else {
        int total = 0;
        for (int j = 0; j < a.nq; j++) total += lens[j];
        for (int i = tid; i < n; i += kThreads) {
            const int j = i / a.K, k = i - j * a.K;
            const int32_t x = lst[i];
            if (x < 0) continue;
            int pos = k;
            for (int jj = 0; jj < a.nq; jj++) {
                if (jj == j) continue;
                const int32_t *l2 = lst + jj * a.K;
                pos += jj < j ? upper_bound(l2, lens[jj], x) : lower_bound(l2, lens[jj], x);
            }
            merged[pos] = x;
        }
        __syncthreads();
        nu = block_compact(
            total, [&](int p) { return p == 0 || merged[p] != merged[p - 1]; },
            [&](int p, int r) { U[r] = merged[p]; }, warp_sums);
        miss = merged;  // merged is dead now
        missidx = lst;  // lists are dead now
    }

    // 3. classify; hits refresh their stamp.  Entries in groups of four per
    // thread, so that their block-table and then hot-map loads are in
    // flight together.
    int nres = 0, nhit = 0, nmiss = 0;
    constexpr int kG = 4;
    for (int i0 = tid; i0 < nu; i0 += kG * kThreads) {
        int32_t u[kG], blk[kG], hs_[kG];
#pragma unroll
        for (int g = 0; g < kG; g++) {
            const int i = i0 + g * kThreads;
            u[g] = i < nu ? U[i] : -1;
            blk[g] = u[g] >= 0 ? bt[u[g] / a.P] : 0;
        }
#pragma unroll
        for (int g = 0; g < kG; g++) hs_[g] = (u[g] >= 0 && blk[g] < 0) ? a.hot_map[hm + u[g]] : -1;
#pragma unroll
        for (int g = 0; g < kG; g++) {
            const int i = i0 + g * kThreads;
            if (i >= nu) continue;
            if (blk[g] >= 0) {
                uslot[i] = -1;
                if (single) rid[i] = blk[g] * a.P + u[g] % a.P;  // one list: U[i] is entry i
                nres++;
            } else if (hs_[g] >= 0) {
                const int32_t s = hs_[g];
                uslot[i] = s;
                a.stamp[sc + s] = step;
                if (single) rid[i] = hb[s / a.P] * a.P + s % a.P;
                nhit++;
            } else {
                uslot[i] = -2;
                nmiss++;
            }
        }
    }
    if (single)
        for (int i = nu + tid; i < n; i += kThreads) rid[i] = -1;  // padding
    int M = 0;
    {
        int tot;  // (hits << 16) | resident: both at most nq * K <= 16384
        block_excl_scan((nhit << 16) | nres, warp_sums, &tot);
        if (tid == 0) {
            atomicAdd(&a.stats[0], (unsigned long long)(tot & 0xFFFF));
            atomicAdd(&a.stats[1], (unsigned long long)(tot >> 16));
        }
    }
    if (__syncthreads_or(nmiss > 0)) {
        M = block_compact(
            nu, [&](int i) { return uslot[i] == -2; },
            [&](int i, int r) {
                miss[r] = U[i];
                missidx[r] = i;
            },
            warp_sums);
    }

    // 4. victims: the Ms smallest (stamp, slot) among slots with stamp < step,
    // Ms = min(M, such slots).  With fewer such slots than misses (possible
    // only with a hot buffer below nq * K rows) the first Ms misses in token
    // order get a slot, the others read nothing, and HS_ERR_CAPACITY is set.
    int served = 0;
    if (M > 0) {
        const uint32_t *stp = a.stamp + sc;
        uint32_t prefix = 0, mask = 0;
        int Ms = M, need = M;
        // Digits above the highest bit set in any candidate stamp are 0 for
        // every candidate and decide nothing: start at the first digit that
        // can differ (stamps are step numbers, so usually the last one).
        // Skipping them also skips histograms whose every count lands in
        // bin 0, where the increments would run one after another.
        uint32_t orv = 0;
        for (int s = tid; s < a.C; s += kThreads) {
            const uint32_t v = stp[s];
            if (v < step) orv |= v;
        }
        orv = __reduce_or_sync(0xffffffffu, orv);
        if ((tid & 31) == 0) warp_sums[tid >> 5] = (int)orv;
        __syncthreads();
        orv = 0;
        for (int w = 0; w < kThreads / 32; w++) orv |= (uint32_t)warp_sums[w];
        __syncthreads();
        const int first = orv == 0 ? 3 : 3 - (31 - __clz(orv)) / 8;
        for (int pass = first; pass < 4; pass++) {
            const int shift = 24 - 8 * pass;
            if (tid < 256) hist[tid] = 0;
            __syncthreads();
            for (int s = tid; s < a.C; s += kThreads) {
                const uint32_t v = stp[s];
                if (v < step && (v & mask) == prefix) atomicAdd(&hist[(v >> shift) & 255u], 1u);
            }
            __syncthreads();
            const int c = tid < 256 ? (int)hist[tid] : 0;
            int tot;
            const int ex = block_excl_scan(c, warp_sums, &tot);
            if (pass == first && tot < Ms) {  // uniform: tot is the block's total
                if (tid == 0) set_error(a.err, HS_ERR_CAPACITY);
                Ms = need = tot;
            }
            if (Ms == 0) break;
            if (tid < 256 && ex < need && need <= ex + c) {
                sel[0] = tid;
                sel[1] = ex;
            }
            __syncthreads();
            prefix |= (uint32_t)sel[0] << shift;
            mask |= 255u << shift;
            need -= sel[1];
            __syncthreads();
        }
        if (Ms > 0) {
            // lt: stamp < S*, eq: stamp == S* (taken lowest slot first, `need` of them)
            const uint32_t S = prefix;
            const int seg = (a.C + kThreads - 1) / kThreads;
            const int lo = min(a.C, tid * seg), hi = min(a.C, lo + seg);
            int lt = 0, eq = 0;
            for (int s = lo; s < hi; s++) {
                const uint32_t v = stp[s];
                lt += v < S;
                eq += (v == S) && (v < step);
            }
            for (int i = tid; i < Ms; i += kThreads) victim[i] = -1;
            __syncthreads();
            int tot;
            const int ex = block_excl_scan((eq << 16) | lt, warp_sums, &tot);
            int lb = ex & 0xFFFF, eb = ex >> 16;
            for (int s = lo; s < hi; s++) {
                const uint32_t v = stp[s];
                if (v < S) {
                    const int pos = lb + min(eb, need);
                    if (pos < Ms) victim[pos] = s;
                    lb++;
                } else if (v == S && v < step) {
                    if (eb < need && lb + eb < Ms) victim[lb + eb] = s;
                    eb++;
                }
            }
            __syncthreads();
            // 5. assignment: i-th miss (ascending token) -> i-th victim (ascending slot)
            for (int i = tid; i < Ms; i += kThreads) {
                const int32_t s = victim[i], u = miss[i];
                if (s < 0 || s >= a.C) {  // cannot happen; never write outside the tables
                    set_error(a.err, HS_ERR_CAPACITY);
                    uslot[missidx[i]] = -3;
                    if (single) rid[missidx[i]] = -1;
                    continue;
                }
                const int32_t old = a.slot_token[sc + s];
                if (old >= 0) a.hot_map[hm + old] = -1;
                a.slot_token[sc + s] = u;
                a.hot_map[hm + u] = s;
                a.stamp[sc + s] = step;
                uslot[missidx[i]] = s;
                if (single) rid[missidx[i]] = hb[s / a.P] * a.P + s % a.P;
                a.miss_tok[(size_t)b * n + i] = u;
                a.miss_slot[(size_t)b * n + i] = s;
            }
        }
        for (int i = Ms + tid; i < M; i += kThreads) {  // misses left without a slot
            uslot[missidx[i]] = -3;
            if (single) rid[missidx[i]] = -1;
        }
        served = Ms;
    }
    if (tid == 0) {
        a.miss_count[b] = served;
        a.req_step[b] = step;
        atomicAdd(&a.stats[2], (unsigned long long)served);
        atomicAdd(&a.stats[3], (unsigned long long)served * a.L * a.R);
    }
    if (single) return;  // every entry's row id is written above
    __syncthreads();

    // 6. row ids: each entry's index in U (from the bitmap's word counts,
    // else a search), its slot, then the row (groups of four per thread,
    // their loads in flight together)
    const uint32_t *bm = (const uint32_t *)(victim + n);
    const int32_t *wpre = (const int32_t *)(bm + a.words);
    for (int i0 = tid; i0 < n; i0 += kG * kThreads) {
        int32_t u[kG], sl[kG], r[kG];
#pragma unroll
        for (int g = 0; g < kG; g++) {
            const int i = i0 + g * kThreads;
            u[g] = i < n ? tk[i] : -1;
        }
#pragma unroll
        for (int g = 0; g < kG; g++) {
            sl[g] = -3;
            if (u[g] >= 0) {
                const int x = u[g];
                const int ui = a.words > 0 ? wpre[x >> 5] + __popc(bm[x >> 5] & ((1u << (x & 31)) - 1u))
                                           : lower_bound(U, nu, x);
                sl[g] = uslot[ui];
            }
        }
#pragma unroll
        for (int g = 0; g < kG; g++) {
            r[g] = -1;
            if (sl[g] == -1)
                r[g] = bt[u[g] / a.P] * a.P + u[g] % a.P;
            else if (sl[g] >= 0)
                r[g] = hb[sl[g] / a.P] * a.P + sl[g] % a.P;
        }
#pragma unroll
        for (int g = 0; g < kG; g++)
            if (i0 + g * kThreads < n) rid[i0 + g * kThreads] = r[g];
    }
}

// Rows of layers [l0, l1) of every miss: 16-byte units over the host link,
// four loads in flight per thread, written to the miss's hot-buffer slot; a
// (gx, B) grid, gx CTAs per request.  Scattered 656-byte rows over the link
// need many SMs' worth of loads in flight: measured at the mixed-residency
// MTP3 workload (64 requests, 776 MB), 608 CTAs move 192 GB/s and 64 CTAs
// (one per request) 189 GB/s, while a flat 24-CTA grid of 512 threads with
// eight loads in flight per thread managed 94 GB/s.
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads) miss_copy_kernel(
    const int32_t *__restrict__ miss_count, const int32_t *__restrict__ miss_tok,
    const int32_t *__restrict__ miss_slot, int n, const int32_t *__restrict__ host_block_table,
    const int32_t *__restrict__ hot_blocks, const uint8_t *__restrict__ host_rows,
    uint8_t *__restrict__ rows, int L, int l0, int l1, int P, int R, int max_pages, int hot_pages,
    int32_t *err) {
    hs::tc::grid_dep_launch();
    hs::tc::grid_dep_wait();  // the miss lists come from the plan kernel
    const int b = blockIdx.y;
    const int M = miss_count[b];
    const int cpr = R / 16, nl = l1 - l0, per_miss = nl * cpr;
    const int64_t total = (int64_t)M * per_miss;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < total;
         i0 += kCopyUnroll * stride) {
        const uint4 *src[kCopyUnroll];
        uint4 *dst[kCopyUnroll];
        uint4 v[kCopyUnroll];
#pragma unroll
        for (int k = 0; k < kCopyUnroll; k++) {
            src[k] = nullptr;
            const int64_t i = i0 + k * stride;
            if (i >= total) continue;
            const int m = (int)(i / per_miss);
            const int rem = (int)(i - (int64_t)m * per_miss);
            const int l = l0 + rem / cpr, c = rem % cpr;
            const int32_t u = miss_tok[(size_t)b * n + m], s = miss_slot[(size_t)b * n + m];
            if (u < 0 || u >= max_pages * P || s < 0 || s >= hot_pages * P) {
                set_error(err, HS_ERR_INVALID_ARG);
                continue;
            }
            const int32_t hblk = host_block_table[(size_t)b * max_pages + u / P];
            if (hblk < 0) {
                set_error(err, HS_ERR_INVALID_ARG);
                continue;
            }
            const int32_t dblk = hot_blocks[(size_t)b * hot_pages + s / P];
            src[k] = (const uint4 *)(host_rows + (((size_t)hblk * L + l) * P + u % P) * R) + c;
            dst[k] = (uint4 *)(rows + (((size_t)dblk * L + l) * P + s % P) * R) + c;
        }
#pragma unroll
        for (int k = 0; k < kCopyUnroll; k++)
            if (src[k]) v[k] = *src[k];
#pragma unroll
        for (int k = 0; k < kCopyUnroll; k++)
            if (src[k]) *dst[k] = v[k];
    }
}

// Bitmap words for the union of several lists: while the bitmap and its
// word counts fit beside the five arrays (rows of up to 262,144 tokens).
int plan_words(const hs_pool *p, int nq) {
    const int words = (p->cfg.max_tokens + 31) / 32;
    return nq > 1 && words <= 8192 ? words : 0;
}

size_t plan_smem(int n, int words) { return (size_t)5 * n * 4 + (size_t)words * 8; }

constexpr size_t kPlanSmemMax = 225 * 1024;  // 227 KB per CTA less the kernel's static arrays

// The block table is staged while it fits beside the rest.
int plan_stage_pages(const hs_pool *p, int n, int words) {
    return plan_smem(n, words) + (size_t)p->max_pages * 4 <= kPlanSmemMax ? p->max_pages : 0;
}

}  // namespace

cudaError_t resolve_setup(const hs_pool *p) {
    const size_t sm = plan_smem(p->nq_max * p->cfg.top_k, plan_words(p, p->nq_max));
    if (sm > kPlanSmemMax) return cudaErrorInvalidValue;
    // each launch asks for what its batch needs, the staged table included
    return cudaFuncSetAttribute(resolve_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kPlanSmemMax);
}

int resolve_kernel_count(const hs_pool *p, int, int) { return p->cfg.host_blocks > 0 ? 2 : 1; }

cudaError_t launch_resolve_plan(const hs_pool *p, const int32_t *topk, int B, int nq,
                                int32_t *row_id, cudaStream_t st) {
    PlanArgs a;
    a.topk = topk;
    a.nq = nq;
    a.K = p->cfg.top_k;
    a.P = p->cfg.page_tokens;
    a.C = p->C;
    a.hot_pages = p->hot_pages;
    a.maxT = p->cfg.max_tokens;
    a.max_pages = p->max_pages;
    a.L = p->cfg.num_mla_layers;
    a.R = p->R;
    a.seq_len = p->d.seq_len;
    a.block_table = p->d.block_table;
    a.hot_map = p->d.hot_map;
    a.slot_token = p->d.slot_token;
    a.stamp = p->d.stamp;
    a.hot_blocks = p->d.hot_blocks;
    a.req_step = p->d.req_step;
    a.miss_count = p->d.miss_count;
    a.miss_tok = p->d.miss_tok;
    a.miss_slot = p->d.miss_slot;
    a.row_id = row_id;
    a.err = p->d.err;
    a.stats = p->d.stats;
    a.words = plan_words(p, nq);
    const int n = nq * a.K;
    a.stage_pages = plan_stage_pages(p, n, a.words);
    {
        PdlLaunch lc(dim3(B), dim3(kThreads), plan_smem(n, a.words) + (size_t)a.stage_pages * 4, st);
        cudaError_t e = cudaLaunchKernelEx(&lc.cfg, resolve_plan_kernel, a);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

// The miss copy of the last plan (its miss lists stay in the pool's workspace
// until the next plan), layers [l0, l1).  ctas = 0: about four CTAs per SM
// over the batch (the copy alone); otherwise about that many CTAs in all (a
// copy beside another kernel, which keeps the other SMs).  priority (0 =
// none) goes to the launch, so that the copy's CTAs take SMs as they free up
// before a lower-priority kernel's.
cudaError_t launch_miss_copy(const hs_pool *p, int B, int nq, cudaStream_t st, int l0, int l1,
                             int ctas, int priority) {
    const int n = nq * p->cfg.top_k;
    if (l1 < 0) l1 = p->cfg.num_mla_layers;
    if (p->cfg.host_blocks > 0) {
        const int want = ctas > 0 ? ctas : 4 * kNumSMs;
        const int gx = (want + B - 1) / B;
        PdlLaunch lc(dim3(gx, B), dim3(kCopyThreads), 0, st);
        if (priority) {
            // beside another kernel: no early launch behind the previous
            // copy (its CTAs would hold SMs while they wait), a high priority
            lc.attrs[0].id = cudaLaunchAttributePriority;
            lc.attrs[0].val.priority = priority;
            lc.cfg.numAttrs = 1;
        }
        cudaError_t e = cudaLaunchKernelEx(&lc.cfg, miss_copy_kernel, (const int32_t *)p->d.miss_count,
                                           (const int32_t *)p->d.miss_tok, (const int32_t *)p->d.miss_slot,
                                           n, (const int32_t *)p->d.host_block_table,
                                           (const int32_t *)p->d.hot_blocks, (const uint8_t *)p->host_dev,
                                           p->d.rows, p->cfg.num_mla_layers, l0, l1, p->cfg.page_tokens,
                                           p->R, p->max_pages, p->hot_pages, p->d.err);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_resolve(const hs_pool *p, const int32_t *topk, int B, int nq, int32_t *row_id,
                           cudaStream_t st) {
    cudaError_t e = launch_resolve_plan(p, topk, B, nq, row_id, st);
    return e == cudaSuccess ? launch_miss_copy(p, B, nq, st) : e;
}

}  // namespace hs
