// Sparse MLA decode on a pair of CTAs that split the latent dimensions
// ("Un contexte d'un million sur huit H200", section "Ce qui se passe":
// attention reads only the K selected latent rows; absorbed-MLA form, the
// 576-dim row is the key and its first 512 dims the value):
//   z = scale * q . row,  out = sum softmax(z) * row[:512],  lse = ln sum exp(z)
//
// One 2-CTA cluster owns one query, 128 heads and a range of the K entries,
// processed in chunks of 128 rows.  CTA r holds nope dims [256 r, 256 r + 256)
// and rope dims [32 r, 32 r + 32) of every row of the chunk and of the 128
// query heads, and computes with heads on the MMA M axis (M = 128):
//   S_r = Q_r R_r^T    (S[head][row] over the CTA's 288 dims; the queries'
//                       nope half is the A operand in tensor memory, the rope
//                       half bf16 x bf16 from shared memory)
//   S   = S_0 + S_1    (each CTA sends the other the partial sums of the 64
//                       heads the other normalises, 16 KB per half chunk,
//                       through distributed shared memory)
//   P   = exp2(S - m)  (CTA r runs the softmax of heads [64 r, 64 r + 64):
//                       one thread per (head, half chunk), so the row maximum
//                       and sum are per-thread; a lazy reference maximum per
//                       head, raised only when a chunk exceeds it by > 2^8)
//   O_r += P V_r       (V_r: the CTA's 256 nope dims, two N = 128 MMAs; the
//                       P rows of the other CTA's heads arrive by a bulk copy)
// TMEM (512 columns): queries' nope half [0,128) (fp16 pairs), S [128,256),
// O [256,512).  Four converter warps load each chunk's rows a chunk ahead
// into registers (16-byte loads of the CTA's half of every row; the rows are
// brought into L2 in bulk beforehand) and write them K-block by K-block into
// 128-byte-swizzled fp16 operand tiles (E4M3 x the row's group scale, the
// scale split into two fp16s) and the rope half, bf16 as it is, into a
// 64-byte-swizzled tile, double buffered by chunk, so that chunk c+1's
// K-blocks are converted while chunk c's P V products run.  (Gathering the
// rows with TMA, four 64-byte row slices per copy, was measured about ten
// times slower to land per chunk than these loads.)
// Warp 0 issues the MMAs, warp 1 owns TMEM and prefetches rows, warps 2-9
// run the exchange, softmax, rescale and epilogue (thread = TMEM lane = head,
// one warp per (lane quarter, half chunk)), warps 10, 11, 14 and 15 convert
// (12 and 13 stay idle, keeping the conversion off the softmax's SM
// sub-partitions).
// Every wait is bounded; on a time-out the kernel records HS_ERR_TIMEOUT,
// skips the remaining work and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "tc.cuh"

namespace hs {
namespace {

constexpr int kRowsPerChunk = 128;
constexpr int kPairHeads = 128;
constexpr int kPairThreads = 512;  // 16 warps (12 and 13 idle, see below)
constexpr int kKbBytes = 16384;    // 128 rows x 64 fp16 (128-byte swizzle)
constexpr float kRescaleLog2 = 8.f;
constexpr float kLog2eP = 1.4426950408889634f;
constexpr float kLn2P = 0.6931471805599453f;
constexpr float kMaxF16P = 65504.f;
constexpr uint32_t kPFullBytes = 2 * 64 * 128 + 64 * 4;  // the peer's P rows + rescale factors
constexpr uint32_t kSrxBytes = 64 * 128 * 4;              // the peer's partial scores of 64 heads

struct PairSmem {
    static constexpr int rn = 0;                              // 2 buffers x 4 K-blocks (fp16)
    static constexpr int pb = rn + 2 * 4 * kKbBytes;          // P: 2 K-blocks (fp16)
    static constexpr int qr = pb + 2 * kKbBytes;              // queries' rope half (bf16, 64-byte swizzle)
    static constexpr int rr = qr + 8192;                      // rows' rope half, 2 buffers (same layout)
    static constexpr int srx = rr + 2 * 8192;                 // received partial S: [32][64] float4
    static constexpr int alpha_rx = srx + 32768;              // [64] peer's rescale factors
    static constexpr int lm_rx = alpha_rx + 256;              // [2][64] peer's l, m
    static constexpr int mx = lm_rx + 512;                    // [2][64] half-chunk maxima
    static constexpr int lsum = mx + 512;                     // [2][64] half-chunk sums
    static constexpr int bars = lsum + 512;
    static constexpr int nbar = 40;
    static constexpr int tslot = bars + nbar * 8;
    static constexpr int bytes = tslot + 16 + 1024;           // + alignment slack
};
static_assert(PairSmem::bytes <= 232448, "pair attention shared memory");

struct PairArgs {
    const __nv_bfloat16 *q;  // [rows][H][576]
    const int32_t *row_id;   // [rows][K]
    const uint8_t *pool;     // block pool base (the rows' scales are read from it)
    int layer, L, P, H, K, splits, kc, max_row;
    float scale_log2;
    __nv_bfloat16 *out;      // [rows][H][512]
    float *lse;
    float *part;             // [rows][H][splits][514]
    int q_ready;
    int32_t *err;
};

// Has the phase with this parity completed?  (test_wait: never suspends the
// thread, so a warp can poll two barriers and take whichever is ready.)
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P1;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, P1;\n\t}"
        : "=r"(ok)
        : "r"(tc::smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same, with acquire at cluster scope (for phases completed by the peer).
__device__ __forceinline__ bool mbar_test_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P1;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 P1, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, P1;\n\t}"
        : "=r"(ok)
        : "r"(tc::smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait by every lane of a warp; true when all lanes saw the phase.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int32_t *err) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(bar, parity, err);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

__device__ __forceinline__ bool warp_wait_cluster(uint64_t *bar, uint32_t parity, int32_t *err) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait_cluster(bar, parity, err);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// OR of a flag over the 256 softmax threads (named barrier 1) or over the
// 128 threads of one CTA's own heads (barrier 2).
__device__ __forceinline__ bool bar_or(uint32_t id, uint32_t count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *(uint32_t *)&v;
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *(uint32_t *)&v;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t e4m3x2_scaled(__nv_fp8x2_storage_t v, __half2 s_hi, __half2 s_lo) {
    const __half2 x = __half2(__nv_cvt_fp8x2_to_halfraw2(v, __NV_E4M3));
    const __half2 y = __hfma2(x, s_hi, __hmul2(x, s_lo));
    return *(const uint32_t *)&y;
}

__device__ __forceinline__ bool bf16x2_beyond_f16(uint32_t w) {
    return (w & 0x7FFFu) > 0x477Fu || ((w >> 16) & 0x7FFFu) > 0x477Fu;
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    return pack_h2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__global__ void __launch_bounds__(kPairThreads, 1)
    attn_pair_kernel(PairArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *rn = smem + PairSmem::rn;
    uint8_t *pb = smem + PairSmem::pb;
    uint8_t *qr = smem + PairSmem::qr;
    uint8_t *rr = smem + PairSmem::rr;
    float4 *srx = (float4 *)(smem + PairSmem::srx);
    float *alpha_rx = (float *)(smem + PairSmem::alpha_rx);
    float *lm_rx = (float *)(smem + PairSmem::lm_rx);
    float *mxs = (float *)(smem + PairSmem::mx);
    float *lss = (float *)(smem + PairSmem::lsum);
    uint64_t *bar = (uint64_t *)(smem + PairSmem::bars);
    uint64_t *kbf = bar;                  // [2][4]: K-block (and, for 0, the rope tile) converted
    uint64_t *kbfree = bar + 8;           // [2][2]: K-blocks 0-1 / 2-3 (and the rope tile) read
    uint64_t *s_full = bar + 24;
    uint64_t *s_free = bar + 25;
    uint64_t *srx_full = bar + 26;        // the peer's partial scores of a chunk arrived
    uint64_t *srx_free = bar + 28;        // the peer has read this CTA's last partial scores
    uint64_t *p_full = bar + 29;
    uint64_t *pb_free = bar + 30;
    uint64_t *o_ready = bar + 31;
    uint64_t *o_done = bar + 32;
    uint64_t *q_full = bar + 33;
    uint64_t *lm_full = bar + 34;
    uint64_t *mma_done = bar + 35;
    uint32_t *tslot = (uint32_t *)(smem + PairSmem::tslot);

    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const uint32_t peer = rank ^ 1u;
    const int split = blockIdx.x >> 1, qrow = blockIdx.y, hg = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k0 = split * a.kc, k1 = min(a.K, k0 + a.kc);
    const int nch = k1 > k0 ? (k1 - k0 + kRowsPerChunk - 1) / kRowsPerChunk : 0;
    const int32_t *ids = a.row_id + (size_t)qrow * a.K;
    const size_t head0 = (size_t)qrow * a.H + (size_t)hg * kPairHeads;  // first head row

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) {
            for (int k = 0; k < 4; k++) tc::mbar_init(&kbf[i * 4 + k], 4);
            for (int k = 0; k < 2; k++) tc::mbar_init(&kbfree[i * 2 + k], 1);
        }
        tc::mbar_init(srx_full, 1);
        tc::mbar_init(s_full, 1);
        tc::mbar_init(s_free, 8);
        tc::mbar_init(srx_free, 4);
        tc::mbar_init(p_full, 1);
        tc::mbar_init(pb_free, 2);
        tc::mbar_init(o_ready, 8);
        tc::mbar_init(o_done, 1);
        tc::mbar_init(q_full, 8);
        tc::mbar_init(lm_full, 1);
        tc::mbar_init(mma_done, 1);
        tc::fence_barrier_init();
        // the first phase of every barrier the peer completes with transaction
        // bytes is armed now, before the peer can send (each later phase is
        // armed by the thread that waited for the phase before it)
        if (nch > 0) {
            tc::mbar_expect_tx(srx_full, kSrxBytes);
            tc::mbar_expect_tx(p_full, kPFullBytes);
            tc::mbar_expect_tx(lm_full, 512);
        }
    }
    if (warp == 1) {
        tc::tmem_alloc(tslot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync();  // both CTAs' barriers exist before any remote arrival
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    tc::grid_dep_launch();
    const uint32_t QN = 0, SC = 128, OC = 256;  // TMEM column bases
    bool ok = true;
    bool range_bad = false;

    if (warp == 0) {
        // ------------------------------------------------------------ MMAs
        tc::grid_dep_wait();
        if (lane == 0 && nch > 0) {
            const uint32_t id_rope = tc::instr_desc(128, 128, 1, 1, 0, 0);  // bf16 x bf16
            const uint32_t id_s = tc::instr_desc(128, 128, 0, 0, 0, 0);     // fp16 (A in TMEM) x fp16
            const uint32_t id_o = tc::instr_desc(128, 128, 0, 0, 0, 1);     // P (K-major) x V (MN-major)
            const uint32_t rn_a = tc::smem_addr(rn), pb_a = tc::smem_addr(pb);
            const uint32_t qr_a = tc::smem_addr(qr), rr_a = tc::smem_addr(rr);
            ok = tc::mbar_wait(q_full, 0, a.err);
            // Issue S and O in the order their inputs arrive: S(sc) K-block by
            // K-block as the converters finish them (after the softmax side has
            // read S(sc-1)), O(oc) as soon as both CTAs' P(oc) is there.  (A
            // fixed S(c+1)-then-O(c) order made O(c), and the P buffer it frees
            // for the next softmax, wait for chunk c+1's conversion.)
            int sc = 0, skb = 0, oc = 0;
            long long t_last = clock64();
            while (ok && oc < nch) {
                bool prog = false;
                if (sc < nch) {
                    const int b = sc & 1;
                    bool go = true;
                    if (skb == 0 && sc >= 1) go = mbar_test(s_free, (sc - 1) & 1);
                    if (go) go = mbar_test(&kbf[b * 4 + skb], (sc >> 1) & 1);
                    if (go) {
                        tc::fence_after_sync();
                        if (skb == 0) {  // the rope tile is converted with K-block 0
#pragma unroll
                            for (int kk = 0; kk < 2; kk++) {
                                const uint64_t ad = tc::smem_desc(qr_a + kk * 32, 16, 512, 4);
                                const uint64_t bd = tc::smem_desc(rr_a + b * 8192 + kk * 32, 16, 512, 4);
                                tc::mma_f16(tmem + SC, ad, bd, id_rope, kk);
                            }
                        }
#pragma unroll
                        for (int kk = 0; kk < 4; kk++) {
                            const uint64_t bd = tc::smem_desc_sw128(rn_a + (b * 4 + skb) * kKbBytes + kk * 32, 16, 1024);
                            tc::mma_f16_tmem_a(tmem + SC, tmem + QN + skb * 32 + kk * 8, bd, id_s, 1);
                        }
                        if (++skb == 4) {
                            tc::mma_commit(s_full);
                            skb = 0;
                            sc++;
                        }
                        prog = true;
                    }
                }
                if (oc < sc && mbar_test(o_ready, oc & 1)) {  // O(oc) += P V
                    const int c = oc, b = c & 1;
                    tc::fence_after_sync();
#pragma unroll
                    for (int half = 0; half < 2; half++) {
#pragma unroll
                        for (int kk = 0; kk < 8; kk++) {
                            const uint64_t ad = tc::smem_desc_sw128(pb_a + (kk >> 2) * kKbBytes + (kk & 3) * 32, 16, 1024);
                            const uint64_t bd = tc::smem_desc_sw128(
                                rn_a + (b * 4 + 2 * half) * kKbBytes + kk * 2048, kKbBytes, 1024);
                            tc::mma_f16(tmem + OC + half * 128, ad, bd, id_o, (c | kk) != 0);
                        }
                        tc::mma_commit(&kbfree[b * 2 + half]);
                    }
                    tc::mma_commit(o_done);
                    // both CTAs may write the next chunk's P (none after the last)
                    if (c + 1 < nch) tc::mma_commit_multicast(pb_free, (uint16_t)0x3);
                    oc++;
                    prog = true;
                }
                if (prog) {
                    t_last = clock64();
                } else if (clock64() - t_last > tc::kWaitCycles) {
                    set_error(a.err, HS_ERR_TIMEOUT);
                    ok = false;
                } else {
                    __nanosleep(20);  // leave the SMSP's issue slots to the other warps
                }
            }
            tc::mma_commit(mma_done);
            tc::mbar_wait(mma_done, 0, a.err);
        }
    } else if (warp == 1) {
        // --------------------------------------------------- L2 prefetch
        // (this CTA 64 of each chunk's 128 rows, all 656 bytes: the peer reads
        // the other half of every row and prefetches the other 64 rows)
        tc::grid_dep_wait();
        auto prefetch = [&](int c) {
#pragma unroll
            for (int i = 0; i < 2; i++) {
                const int k = k0 + c * kRowsPerChunk + 64 * (int)rank + 32 * i + lane;
                const int32_t id = (c < nch && k < k1) ? ids[k] : -1;
                if (id >= 0 && id < a.max_row)
                    tc::prefetch_l2(a.pool + (((size_t)(id / a.P) * a.L + a.layer) * a.P + id % a.P) * 656, 656);
            }
        };
        // in chunk order: the first chunks' rows arrive first
        for (int c = 0; c < nch; c++) prefetch(c);
    } else if (warp == 12 || warp == 13) {
        // idle: a warp's SM sub-partition is warp % 4, and sub-partitions 0
        // and 1 run the softmax of this CTA's heads (TMEM lanes 0-63 or
        // 64-127 are read from two sub-partitions only), so the converters
        // are warps 10, 11, 14 and 15, on sub-partitions 2 and 3 (measured
        // 354.9 -> 344.7 us at 64 x 4 queries against warps 10-13)
    } else if (warp >= 10) {
        // ------------------------------------------------------ converters
        // Thread ct owns rows ct/4 + 32 i (i < 4) and the 16-byte slice ct % 4
        // of each row's 64 bytes in every nope K-block of this CTA's half and
        // of its rope half: 16 + 4 loads of 16 bytes and 4 of the rows' two
        // group scales per chunk, issued a chunk ahead into registers.
        tc::grid_dep_wait();
        const int ct = warp < 14 ? threadIdx.x - 320 : threadIdx.x - 384;  // 0..127
        const int part = ct & 3;
        uint4 raw[4][4], rope[4];
        float2 sg[4];
        auto load = [&](int c) {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int k = k0 + c * kRowsPerChunk + (ct >> 2) + 32 * i;
                int32_t id = (c < nch && k < k1) ? ids[k] : -1;
                if (id >= a.max_row) {
                    set_error(a.err, HS_ERR_INDEX_RANGE);
                    id = -1;
                }
                if (id < 0) {
#pragma unroll
                    for (int kb = 0; kb < 4; kb++) raw[kb][i] = make_uint4(0, 0, 0, 0);
                    rope[i] = make_uint4(0, 0, 0, 0);
                    sg[i] = make_float2(0.f, 0.f);
                    continue;
                }
                const uint8_t *row = a.pool + (((size_t)(id / a.P) * a.L + a.layer) * a.P + id % a.P) * 656;
#pragma unroll
                for (int kb = 0; kb < 4; kb++) raw[kb][i] = tc::ld_nc16(row + 256 * rank + 64 * kb + 16 * part);
                rope[i] = tc::ld_nc16(row + 528 + 64 * rank + 16 * part);
                const uint2 w = tc::ld_nc8(row + 512 + 8 * rank);
                sg[i] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
            }
        };
        load(0);
        for (int c = 0; c < nch && ok; c++) {
            const int b = c & 1;
            for (int kb = 0; kb < 4; kb++) {
                if (c >= 2 && (kb & 1) == 0 &&
                    !(ok = warp_wait(&kbfree[b * 2 + (kb >> 1)], ((c - 2) >> 1) & 1, a.err)))
                    break;
                if (kb == 0) {  // the rope half: bf16 as it is, into its 64-byte-swizzled tile
                    uint8_t *rt = rr + b * 8192;
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        *(uint4 *)(rt + tc::sw64_offset((ct >> 2) + 32 * i, part)) = rope[i];
                }
                uint8_t *dst = rn + (b * 4 + kb) * kKbBytes;
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int r = (ct >> 2) + 32 * i;
                    const float scl = (kb >> 1) ? sg[i].y : sg[i].x;
                    range_bad |= 448.f * fabsf(scl) > kMaxF16P;
                    const __half s_hi = __float2half_rn(scl);
                    const __half2 shi2 = __half2half2(s_hi);
                    const __half2 slo2 = __half2half2(__float2half_rn(scl - __half2float(s_hi)));
                    const __nv_fp8x2_storage_t *pp = (const __nv_fp8x2_storage_t *)&raw[kb][i];
                    uint32_t h[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) h[e] = e4m3x2_scaled(pp[e], shi2, slo2);
                    *(uint4 *)(dst + tc::sw128_offset(r, 2 * part)) = make_uint4(h[0], h[1], h[2], h[3]);
                    *(uint4 *)(dst + tc::sw128_offset(r, 2 * part + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
                }
                tc::fence_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&kbf[b * 4 + kb]);
            }
            if (ok) load(c + 1);  // the registers are free: the next chunk's rows
        }
    } else {
        // ------------------------------- exchange, softmax, rescale, output
        const int sp = warp & 3, ch = (warp - 2) >> 2;
        const int h = 32 * sp + lane;                  // head = TMEM lane
        const bool own = (sp >> 1) == (int)rank;       // this CTA normalises heads [64 rank, +64)
        const int ho = h - 64 * (int)rank;             // index among own heads
        const int hp = h - 64 * (int)peer;             // index among the peer's heads
        const uint32_t lane_base = tmem + ((uint32_t)(32 * sp) << 16);
        // queries: the nope half of head h (dims 256 rank + 128 ch ..) -> TMEM,
        // fp16 pairs; the rope half of every head -> the 64-byte-swizzled tile
        const __nv_bfloat16 *qh = a.q + (head0 + h) * kLatent;
        auto load_q = [&]() {
            const uint4 *src = (const uint4 *)(qh + 256 * rank + 128 * ch);
#pragma unroll
            for (int half = 0; half < 2; half++) {
                uint32_t v[32];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const uint4 w = src[half * 8 + i];
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        range_bad |= bf16x2_beyond_f16(ws[e]);
                        v[4 * i + e] = bf16x2_to_f16x2(ws[e]);
                    }
                }
                tc::tmem_st32(lane_base + QN + 64 * ch + 32 * half, v);
            }
            const int t = threadIdx.x - 64;  // 0..255
#pragma unroll
            for (int i = 0; i < 2; i++) {
                const int unit = t + 256 * i, hh = unit >> 2, part = unit & 3;
                const uint4 w = *(const uint4 *)(a.q + (head0 + hh) * kLatent + 512 + 32 * rank + 8 * part);
                *(uint4 *)(qr + tc::sw64_offset(hh, part)) = w;
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc::fence_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(q_full);
        };
        if (a.q_ready) load_q();
        tc::grid_dep_wait();
        if (!a.q_ready) load_q();

        float mref = -INFINITY, lpart = 0.f;
        const uint32_t srx_peer = tc::mapa(tc::smem_addr(srx), peer);
        const uint32_t srx_full_peer = tc::mapa(tc::smem_addr(srx_full), peer);
        const uint32_t srx_free_peer = tc::mapa(tc::smem_addr(srx_free), peer);
        const uint32_t p_full_peer = tc::mapa(tc::smem_addr(p_full), peer);
        const uint32_t alpha_peer = tc::mapa(tc::smem_addr(alpha_rx), peer);
        // the warp that waits for a transfer barrier also arms its next phase
        const bool p_armer = !own && ch == 0 && sp == 2 * (int)peer && lane == 0;
        const bool s_armer = own && sp == 2 * (int)rank && ch == 0 && lane == 0;
        // a sender warp's handling of chunk cc's arrival from the peer: its P
        // rows and rescale factors; rescale this CTA's O rows of the peer's
        // heads when needed, then let the MMA warp run O(cc)
        auto sender_finish = [&](int cc) -> bool {
            if (!warp_wait_cluster(p_full, cc & 1, a.err)) return false;
            if (p_armer && cc + 1 < nch) tc::mbar_expect_tx(p_full, kPFullBytes);
            const float al = alpha_rx[hp];
            // the warp rescales together (TMEM loads and stores are warp-wide);
            // before chunk 0's P V there is nothing to scale
            if (__any_sync(0xffffffffu, al != 1.f) && cc >= 1) {
                if (!warp_wait(o_done, (cc - 1) & 1, a.err)) return false;
                tc::fence_after_sync();
#pragma unroll 1
                for (int q = 0; q < 8; q++) {
                    float o[16];
                    const uint32_t ta = lane_base + OC + 128 * ch + 16 * q;
                    tc::tmem_ld16(ta, o);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; i++) o[i] *= al;
                    tc::tmem_st16(ta, o);
                }
                tc::tmem_st_wait();
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(o_ready);
            return true;
        };
        int32_t idn[2];  // an own warp's row ids of the chunk it processes next
#pragma unroll
        for (int w2 = 0; w2 < 2; w2++) {
            const int k = k0 + 64 * ch + 32 * w2 + lane;
            idn[w2] = (own && nch > 0 && k < k1) ? ids[k] : -1;
        }
        for (int c = 0; c < nch && ok; c++) {
            const uint32_t sbase = lane_base + SC + 64 * ch;
            if (!own) {
                // ---- a sender warp has two things to do per chunk, in the
                // order their inputs arrive: send S(c)'s partial sums of the
                // peer's heads (once S(c) is done and the peer has read the
                // last chunk's), and complete chunk c-1 with the peer's P rows
                // (which lets the MMA warp issue O(c-1); O(c-1) frees the P
                // buffer that the next softmax writes).  Waiting for either
                // one first put the other on the chunk's critical path
                // (measured 9.3-10 K cycles per chunk).
                bool need_fin = c >= 1, need_send = true;
                const long long t0 = clock64();
                while (ok && (need_fin || need_send)) {
                    int rdy = 0;  // lane 0's view, made the warp's
                    if (lane == 0) {
                        if (need_fin && mbar_test_cluster(p_full, (c - 1) & 1)) rdy |= 1;
                        if (need_send && mbar_test(s_full, c & 1)) rdy |= 2;
                        if (!rdy && clock64() - t0 > tc::kWaitCycles) rdy = 4;
                    }
                    rdy = __shfl_sync(0xffffffffu, rdy, 0);
                    if (rdy & 1) {
                        ok = sender_finish(c - 1);
                        need_fin = false;
                    } else if (rdy & 2) {
                        tc::fence_after_sync();
                        // after the peer has read the last chunk's partial sums
                        if (c >= 1 && !(ok = warp_wait_cluster(srx_free, (c - 1) & 1, a.err))) break;
#pragma unroll
                        for (int q4 = 0; q4 < 4; q4++) {
                            float v[16];
                            tc::tmem_ld16(sbase + 16 * q4, v);
                            tc::tmem_ld_wait();
#pragma unroll
                            for (int j4 = 0; j4 < 4; j4++) {
                                const uint4 w = make_uint4(__float_as_uint(v[4 * j4]), __float_as_uint(v[4 * j4 + 1]),
                                                           __float_as_uint(v[4 * j4 + 2]), __float_as_uint(v[4 * j4 + 3]));
                                tc::st_async_v4(srx_peer + (uint32_t)(((16 * ch + 4 * q4 + j4) * 64 + hp) * 16), w,
                                                srx_full_peer);
                            }
                        }
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(s_free);
                        need_send = false;
                    } else if (rdy & 4) {
                        if (lane == 0) set_error(a.err, HS_ERR_TIMEOUT);
                        ok = false;
                    } else {
                        __nanosleep(20);
                    }
                }
                continue;
            }
            // validity of this warp's 64 rows; the next chunk's ids load now
            // and arrive while this chunk runs
            uint32_t vm[2];
#pragma unroll
            for (int w2 = 0; w2 < 2; w2++) {
                vm[w2] = __ballot_sync(0xffffffffu, idn[w2] >= 0 && idn[w2] < a.max_row);
                const int k = k0 + (c + 1) * kRowsPerChunk + 64 * ch + 32 * w2 + lane;
                idn[w2] = (c + 1 < nch && k < k1) ? ids[k] : -1;
            }
            if (!(ok = warp_wait(s_full, c & 1, a.err))) {
                bar_or(2, 128, true);  // the partners leave at their next barrier
                break;
            }
            tc::fence_after_sync();
            {
                float v[64];
#pragma unroll
                for (int q4 = 0; q4 < 4; q4++) tc::tmem_ld16(sbase + 16 * q4, v + 16 * q4);
                tc::tmem_ld_wait();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(s_free);
                // ---- receive the peer's partial sums of these heads
                if (!(ok = warp_wait_cluster(srx_full, c & 1, a.err))) {
                    bar_or(2, 128, true);
                    break;
                }
                if (s_armer && c + 1 < nch) tc::mbar_expect_tx(srx_full, kSrxBytes);
                float lmax = -INFINITY;
#pragma unroll
                for (int j4 = 0; j4 < 16; j4++) {
                    const float4 pv = srx[(16 * ch + j4) * 64 + ho];
                    const float pp[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int j = 4 * j4 + e;
                        const bool valid = (vm[j >> 5] >> (j & 31)) & 1u;
                        v[j] = valid ? (v[j] + pp[e]) * a.scale_log2 : -INFINITY;
                        lmax = fmaxf(lmax, v[j]);
                    }
                }
                __syncwarp();
                // srx may take the next chunk (relaxed: the values read are already used)
                if (lane == 0) tc::mbar_arrive_remote_relaxed(srx_free_peer);
                mxs[ch * 64 + ho] = lmax;
                if (bar_or(2, 128, false)) {  // a partner timed out
                    ok = false;
                    break;
                }
                const float cm = fmaxf(lmax, mxs[(1 - ch) * 64 + ho]);
                float mnew = mref, al = 1.f;
                if (cm > -INFINITY && (mref == -INFINITY || cm > mref + kRescaleLog2)) {
                    mnew = cm;
                    al = mref == -INFINITY ? 0.f : ex2(mref - mnew);
                }
                // P(c) may overwrite P(c-1) once O(c-1) is done in both CTAs
                if (c >= 1 && !(ok = warp_wait_cluster(pb_free, (c - 1) & 1, a.err))) {
                    bar_or(2, 128, true);
                    break;
                }
                float psum = 0.f;
                uint8_t *prow = pb + ch * kKbBytes;
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int j = 8 * q + 2 * e;
                        const float p0 = mnew == -INFINITY ? 0.f : ex2(v[j] - mnew);
                        const float p1 = mnew == -INFINITY ? 0.f : ex2(v[j + 1] - mnew);
                        psum += p0 + p1;
                        pk[e] = pack_h2(p0, p1);
                    }
                    *(uint4 *)(prow + tc::sw128_offset(h, q)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                lpart = lpart * al + psum;
                mref = mnew;
                if (ch == 0) tc::st_async_b32(alpha_peer + 4 * ho, __float_as_uint(al), p_full_peer);
                if (__any_sync(0xffffffffu, al != 1.f) && c >= 1) {  // (warp-wide, as above)
                    if (!(ok = warp_wait(o_done, (c - 1) & 1, a.err))) {
                        bar_or(2, 128, true);
                        break;
                    }
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int q = 0; q < 8; q++) {
                        float o[16];
                        const uint32_t ta = lane_base + OC + 128 * ch + 16 * q;
                        tc::tmem_ld16(ta, o);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; i++) o[i] *= al;
                        tc::tmem_st16(ta, o);
                    }
                    tc::tmem_st_wait();
                }
                tc::fence_async_smem();  // P is read by the tensor core (async proxy)
                tc::fence_before_sync();
                // every own-head P row of this chunk is written: send them to the peer
                if (bar_or(2, 128, false)) {
                    ok = false;
                    break;
                }
                if (sp == 2 * (int)rank && ch == 0 && lane == 0) {
#pragma unroll
                    for (int kbp = 0; kbp < 2; kbp++) {
                        const uint32_t off = kbp * kKbBytes + 64 * rank * 128;
                        tc::bulk_s2s(tc::mapa(tc::smem_addr(pb + off), peer), pb + off, 8192, p_full_peer);
                    }
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(o_ready);
            }
        }
        if (!own && ok && nch > 0) ok = sender_finish(nch - 1);
        // ------------------------------------------------------------ output
        // own heads: l = the two half-chunk sums, m = the reference maximum;
        // the peer's heads: (l, m) from the peer
        if (ok && own) {
            lss[ch * 64 + ho] = lpart;
            if (bar_or(2, 128, false)) ok = false;
        }
        float l = 0.f, m = -INFINITY;
        if (own) {
            if (ok) {
                l = lss[ho] + lss[64 + ho];
                m = mref;
                if (ch == 0) {
                    const uint32_t lm_peer = tc::mapa(tc::smem_addr(lm_rx), peer);
                    const uint32_t lm_full_peer = tc::mapa(tc::smem_addr(lm_full), peer);
                    tc::st_async_b32(lm_peer + 4 * ho, __float_as_uint(l), lm_full_peer);
                    tc::st_async_b32(lm_peer + 256 + 4 * ho, __float_as_uint(m), lm_full_peer);
                }
            }
        } else {
            if (ok && nch > 0) {
                ok = warp_wait_cluster(lm_full, 0, a.err);
                l = lm_rx[hp];
                m = lm_rx[64 + hp];
            }
        }
        bool fin = ok && (nch == 0 || warp_wait(o_done, (nch - 1) & 1, a.err));
        tc::fence_after_sync();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int dbase = 256 * (int)rank + 128 * ch;
        if (a.splits == 1) {
            __nv_bfloat16 *dst = a.out + (head0 + h) * kNope + dbase;
#pragma unroll 1
            for (int q = 0; q < 8; q++) {
                float o[16];
                if (fin && nch > 0) {
                    tc::tmem_ld16(lane_base + OC + 128 * ch + 16 * q, o);
                    tc::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 16; i++) o[i] = 0.f;
                }
                uint4 w0, w1;
                w0.x = pack_bf2(o[0] * inv, o[1] * inv);
                w0.y = pack_bf2(o[2] * inv, o[3] * inv);
                w0.z = pack_bf2(o[4] * inv, o[5] * inv);
                w0.w = pack_bf2(o[6] * inv, o[7] * inv);
                w1.x = pack_bf2(o[8] * inv, o[9] * inv);
                w1.y = pack_bf2(o[10] * inv, o[11] * inv);
                w1.z = pack_bf2(o[12] * inv, o[13] * inv);
                w1.w = pack_bf2(o[14] * inv, o[15] * inv);
                *(uint4 *)(dst + 16 * q) = w0;
                *(uint4 *)(dst + 16 * q + 8) = w1;
            }
            if (own && ch == 0 && a.lse) a.lse[head0 + h] = l > 0.f ? (m + log2f(l)) * kLn2P : -INFINITY;
        } else {
            float *rec = a.part + ((head0 + h) * a.splits + split) * (kNope + 2);
#pragma unroll 1
            for (int q = 0; q < 8; q++) {
                float o[16];
                if (fin && nch > 0) {
                    tc::tmem_ld16(lane_base + OC + 128 * ch + 16 * q, o);
                    tc::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 16; i++) o[i] = 0.f;
                }
#pragma unroll
                for (int i = 0; i < 16; i += 2)  // records are 514 floats: 8-byte aligned only
                    *(float2 *)(rec + dbase + 16 * q + i) = make_float2(o[i], o[i + 1]);
            }
            if (own && ch == 0) {
                rec[kNope] = l > 0.f ? m : -INFINITY;
                rec[kNope + 1] = l;
            }
        }
    }
    if (range_bad) set_error(a.err, HS_ERR_RANGE);
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync();  // no transfer into this CTA's shared memory is in flight
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool pair_eligible(const hs_pool *p) {
    return p->cfg.row_fmt == HS_ROW_E4M3_656 && p->cfg.mla_heads % kPairHeads == 0;
}

// Row ranges per query for the pair kernel: one 2-CTA cluster per (query,
// 128 heads, range), one CTA per SM.  Cost in chunk times: waves x (chunks
// per range + about three of start-up) + one for the combine pass.
int pair_splits(const hs_pool_config &c, int rows) {
    const int chunks = (c.top_k + kRowsPerChunk - 1) / kRowsPerChunk;
    const int pairs = rows * (c.mla_heads / kPairHeads);
    const int slots = kNumSMs / 2;
    int best = 1;
    long best_cost = -1;
    for (int s = 1; s <= chunks && s <= kMaxSplits; s++) {
        const long cps = (chunks + s - 1) / s;
        const long waves = ((long)pairs * s + slots - 1) / slots;
        const long cost = waves * (cps + 3) + (s > 1 ? 1 : 0);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    const int kc = ((c.top_k + best - 1) / best + kRowsPerChunk - 1) / kRowsPerChunk * kRowsPerChunk;
    return (c.top_k + kc - 1) / kc;
}

cudaError_t pair_setup(const hs_pool *) {
    return cudaFuncSetAttribute(attn_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PairSmem::bytes);
}

cudaError_t launch_pair_attention(const hs_pool *p, int layer, const void *q, const int32_t *row_id, int B,
                                  int nq, float scale, void *out, float *lse, cudaStream_t st, bool q_ready, bool pdl) {
    const int rows = B * nq, K = p->cfg.top_k;
    const int splits = pair_splits(p->cfg, rows);
    PairArgs a;
    a.q = (const __nv_bfloat16 *)q;
    a.row_id = row_id;
    a.pool = p->d.rows;
    a.layer = layer;
    a.L = p->cfg.num_mla_layers;
    a.P = p->cfg.page_tokens;
    a.H = p->cfg.mla_heads;
    a.K = K;
    a.splits = splits;
    a.kc = ((K + splits - 1) / splits + kRowsPerChunk - 1) / kRowsPerChunk * kRowsPerChunk;
    a.max_row = (int)(p->cfg.gpu_blocks * p->cfg.page_tokens);
    a.scale_log2 = scale * kLog2eP;
    a.out = (__nv_bfloat16 *)out;
    a.lse = lse;
    a.part = p->d.attn_part;
    a.q_ready = q_ready;
    a.err = p->d.err;
    dim3 grid(2 * splits, rows, a.H / kPairHeads);
    PdlLaunch lc(grid, dim3(kPairThreads), PairSmem::bytes, st, dim3(2, 1, 1), pdl);
    return cudaLaunchKernelEx(&lc.cfg, attn_pair_kernel, a);
}

}  // namespace hs
