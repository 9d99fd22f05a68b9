// Host side of libhs: pool carving, request lifecycle, introspection and the
// orchestration of one decode step.  Nothing here runs on the decode path
// except hs_step's enqueue sequence, which makes no host decision that
// depends on device data.
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "hs_internal.h"

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
        else
            cudaGetLastError();
    }
    return fn;
}

// 2-D view of the key slab: rows = max_requests * max_tokens, 128 bytes
// each; one TMA box = 128 rows x 128 bytes with the 128-byte swizzle the
// tensor core reads.
bool make_key_map(hs_pool *p) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t gdim[2] = {128, (cuuint64_t)p->cfg.max_requests * (cuuint64_t)p->cfg.max_tokens};
    cuuint64_t gstride[1] = {128};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(&p->key_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, p->d.idx_keys, gdim, gstride,
                     box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

constexpr size_t kAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Carver {
    size_t off = 0;
    size_t take(size_t bytes) {
        size_t o = round_up(off, kAlign);
        off = o + round_up(bytes, 16);
        return o;
    }
};

bool valid_config(const hs_pool_config *c) {
    if (!c) return false;
    if (c->max_requests <= 0 || c->max_tokens <= 0 || c->page_tokens <= 0) return false;
    if (c->top_k <= 0 || c->num_spec < 0 || c->num_spec > 7) return false;
    if (c->tail_tokens < 0 || c->num_mla_layers <= 0 || c->mla_heads <= 0) return false;
    if (c->idx_heads <= 0 || c->idx_dim <= 0) return false;
    if (c->row_fmt != HS_ROW_E4M3_656 && c->row_fmt != HS_ROW_F32_2304) return false;
    if (c->idx_fmt != HS_IDX_E4M3 && c->idx_fmt != HS_IDX_F32) return false;
    if (c->gpu_blocks < 0 || c->host_blocks < 0) return false;
    if (c->gpu_blocks > INT32_MAX || c->host_blocks > INT32_MAX) return false;
    // device row ids are int32; the attention addresses a row by its index in
    // row units of the pool, a uint32
    if (c->gpu_blocks * c->page_tokens > INT32_MAX) return false;
    if (c->gpu_blocks * c->page_tokens * c->num_mla_layers > (int64_t)UINT32_MAX) return false;
    if (c->idx_fmt == HS_IDX_E4M3 && c->idx_dim % 16 != 0) return false;
    if (c->mla_heads % 8 != 0) return false;
    const int nq = c->num_spec + 1;
    const int64_t C = c->hot_rows ? c->hot_rows : (int64_t)(c->num_spec + 2) * c->top_k;
    // below nq * top_k rows a step may find fewer free slots than misses: it
    // reports HS_ERR_CAPACITY and serves what fits
    if (C % c->page_tokens != 0 || C < (int64_t)c->top_k) return false;
    if ((int64_t)nq * c->top_k > 16384) return false;  // resolve keeps the union in smem
    if (C > 16384) return false;
    return true;
}

struct Derived {
    int R, nq, C, hot_pages, max_pages, esize, nchunks;
    int64_t score_stride;
    size_t attn_part_floats;
};

Derived derive(const hs_pool_config *c) {
    Derived d;
    d.R = c->row_fmt == HS_ROW_E4M3_656 ? 656 : 2304;
    d.nq = c->num_spec + 1;
    d.C = c->hot_rows ? c->hot_rows : (c->num_spec + 2) * c->top_k;
    d.hot_pages = d.C / c->page_tokens;
    d.max_pages = (c->max_tokens + c->page_tokens - 1) / c->page_tokens;
    d.esize = c->idx_fmt == HS_IDX_E4M3 ? 1 : 4;
    d.score_stride = (int64_t)round_up((size_t)c->max_tokens, 64);
    d.nchunks = (c->max_tokens + hs::kTopkChunk - 1) / hs::kTopkChunk;
    // split-K partials of the attention (only used while one launch cannot
    // fill the GPU without splitting the K rows)
    d.attn_part_floats = hs::attention_partial_floats(c);
    return d;
}

hs_layout carve(const hs_pool_config *c, const Derived &d, size_t *extra_offs /*[16]*/) {
    Carver cv;
    hs_layout L;
    memset(&L, 0, sizeof L);
    const size_t maxR = c->max_requests, maxT = c->max_tokens;
    L.rows = cv.take((size_t)c->gpu_blocks * c->num_mla_layers * c->page_tokens * d.R);
    L.idx_keys = cv.take(maxR * maxT * c->idx_dim * d.esize);
    L.idx_scale = cv.take(maxR * maxT * 4);
    L.block_table = cv.take(maxR * d.max_pages * 4);
    L.host_block_table = cv.take(maxR * d.max_pages * 4);
    L.hot_map = cv.take(maxR * maxT * 4);
    L.slot_token = cv.take(maxR * d.C * 4);
    L.stamp = cv.take(maxR * d.C * 4);
    L.hot_blocks = cv.take(maxR * d.hot_pages * 4);
    L.seq_len = cv.take(maxR * 4);
    L.req_step = cv.take(maxR * 4);
    const size_t rows = maxR * d.nq;
    extra_offs[0] = cv.take(16);                                      // err
    extra_offs[1] = cv.take(4 * 8);                                   // stats
    extra_offs[2] = cv.take(rows * d.score_stride * 4);               // scores
    extra_offs[3] = cv.take(rows * sizeof(hs::TopkRowState));         // topk state
    extra_offs[4] = cv.take(rows * hs::kTopkBins * 4);                // topk hist
    extra_offs[5] = cv.take(rows * (size_t)d.nchunks * 2 * 4);        // topk chunk counts
    extra_offs[6] = cv.take(maxR * 4);                                // miss count
    extra_offs[7] = cv.take(maxR * (size_t)d.nq * c->top_k * 4);      // miss tok
    extra_offs[8] = cv.take(maxR * (size_t)d.nq * c->top_k * 4);      // miss slot
    extra_offs[9] = cv.take(d.attn_part_floats * 4 + 16);             // attention partials
    extra_offs[10] = c->top_k <= hs::kTopkSampledMaxK                 // top-K candidates
                         ? cv.take(rows * (size_t)hs::kTopkCandCap * 8)
                         : 0;
    L.row_bytes = d.R;
    L.max_pages = d.max_pages;
    L.hot_rows = d.C;
    L.total = round_up(cv.off, kAlign);
    return L;
}

hs_status cuda_status(cudaError_t e) { return e == cudaSuccess ? HS_OK : HS_ERR_CUDA; }

bool req_ok(const hs_pool *p, int32_t req) {
    return p && req >= 0 && req < p->cfg.max_requests;
}

// Upload one request's block-table rows and hot-block list from the mirrors.
cudaError_t upload_tables(hs_pool *p, int32_t req, cudaStream_t st) {
    const size_t mp = p->max_pages;
    cudaError_t e = cudaMemcpyAsync(p->d.block_table + req * mp, p->block_table.data() + req * mp,
                                    mp * 4, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyAsync(p->d.host_block_table + req * mp, p->host_block_table.data() + req * mp,
                        mp * 4, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return e;
    const size_t hp = p->hot_pages;
    e = cudaMemcpyAsync(p->d.hot_blocks + req * hp, p->hot_blocks.data() + req * hp, hp * 4,
                        cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return e;
    return cudaMemcpyAsync(p->d.seq_len + req, p->seq_len.data() + req, 4, cudaMemcpyHostToDevice,
                           st);
}

// Reset the hot-buffer state of one request: no token held, stamps 0, step 0.
cudaError_t reset_hot(hs_pool *p, int32_t req, cudaStream_t st) {
    const size_t maxT = p->cfg.max_tokens, C = p->C;
    cudaError_t e = cudaMemsetAsync(p->d.hot_map + req * maxT, 0xFF, maxT * 4, st);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(p->d.slot_token + req * C, 0xFF, C * 4, st);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(p->d.stamp + req * C, 0, C * 4, st);
    if (e != cudaSuccess) return e;
    return cudaMemsetAsync(p->d.req_step + req, 0, 4, st);
}

int first_tail_page(const hs_pool *p, int mode, int64_t N) {
    const int P = p->cfg.page_tokens;
    if (mode == HS_FULL) return 0;
    if (mode == HS_ZERO) return INT32_MAX;
    int64_t s = N - p->cfg.tail_tokens;
    if (s < 0) s = 0;
    return (int)(s / P);
}

size_t block_bytes(const hs_pool *p) {
    return (size_t)p->cfg.num_mla_layers * p->cfg.page_tokens * p->R;
}

// Device->host copies of whole blocks on `st` (the copy engine), given as
// (GPU block, host block) pairs; runs of neighbouring pairs go as one copy.
cudaError_t copy_blocks_to_host(hs_pool *p, const std::vector<std::pair<int32_t, int32_t>> &pairs,
                                cudaStream_t st) {
    const size_t bb = block_bytes(p);
    cudaError_t e = cudaSuccess;
    for (size_t i = 0; i < pairs.size() && e == cudaSuccess;) {
        size_t j = i + 1;
        while (j < pairs.size() && pairs[j].first == pairs[j - 1].first + 1 &&
               pairs[j].second == pairs[j - 1].second + 1)
            j++;
        e = cudaMemcpyAsync(p->host_base + (size_t)pairs[i].second * bb,
                            p->d.rows + (size_t)pairs[i].first * bb, (j - i) * bb,
                            cudaMemcpyDeviceToHost, st);
        i = j;
    }
    return e;
}

// The pages of `req` listed in `pages` are about to give their GPU block
// back: on `st`, write the host copy of those that have none, and order `st`
// after the pre-copies of the others (a device-side wait, no host wait).
cudaError_t secure_host_copies(hs_pool *p, int32_t req, const std::vector<int> &pages,
                               cudaStream_t st) {
    const size_t mp = p->max_pages;
    const int32_t *bt = p->block_table.data() + req * mp;
    const int32_t *hbt = p->host_block_table.data() + req * mp;
    uint8_t *ok = p->host_ok.data() + req * mp;
    std::vector<std::pair<int32_t, int32_t>> pairs;
    bool wait = false;
    for (int pg : pages) {
        if (ok[pg]) wait = true;
        else pairs.push_back({bt[pg], hbt[pg]});
    }
    cudaError_t e = cudaSuccess;
    if (wait && p->precopy_pending) e = cudaStreamWaitEvent(st, p->precopy_ev, 0);
    if (e == cudaSuccess) e = copy_blocks_to_host(p, pairs, st);
    if (e == cudaSuccess)
        for (int pg : pages) ok[pg] = 1;
    return e;
}

void forget_policy(hs_pool *p, int32_t req) {
    auto &v = p->policy_flipped;
    for (size_t i = 0; i < v.size(); i++)
        if (v[i] == req) {
            v.erase(v.begin() + i);
            return;
        }
}

int resident_pages(const hs_pool *p, int32_t req) {
    const size_t mp = p->max_pages;
    const int32_t *bt = p->block_table.data() + req * mp;
    const int npages = (int)((p->seq_len[req] + p->cfg.page_tokens - 1) / p->cfg.page_tokens);
    int n = 0;
    for (int pg = 0; pg < npages; pg++) n += bt[pg] >= 0;
    return n;
}

// GPU blocks request `req` would hold in `mode` at its current length.
int64_t blocks_in_mode(const hs_pool *p, int32_t req, int mode) {
    const int P = p->cfg.page_tokens;
    const int64_t N = p->seq_len[req];
    const int npages = (int)((N + P - 1) / P);
    const int tail0 = first_tail_page(p, mode, N);
    const int64_t res = std::max(0, npages - std::min(tail0, npages));
    return res + (mode == HS_FULL ? 0 : p->hot_pages);
}

}  // namespace

extern "C" {

int32_t hs_abi_version(void) { return 106; }

const char *hs_status_string(hs_status s) {
    switch (s) {
        case HS_OK: return "ok";
        case HS_ERR_INVALID_ARG: return "invalid argument";
        case HS_ERR_ARENA_TOO_SMALL: return "arena too small";
        case HS_ERR_CAPACITY: return "capacity exhausted (GPU blocks or hot buffer)";
        case HS_ERR_HOST_POOL_FULL: return "pinned host pool full";
        case HS_ERR_INDEX_RANGE: return "selected index outside the request";
        case HS_ERR_TIMEOUT: return "bounded device wait ran out";
        case HS_ERR_CUDA: return "CUDA runtime error";
        case HS_ERR_RANGE: return "value beyond the fp16 range of the tensor-core attention";
    }
    return "unknown status";
}

hs_status hs_pool_required_bytes(const hs_pool_config *cfg, size_t *dev_bytes,
                                 size_t *host_bytes) {
    if (!valid_config(cfg) || !dev_bytes || !host_bytes) return HS_ERR_INVALID_ARG;
    Derived d = derive(cfg);
    size_t extra[16];
    hs_layout L = carve(cfg, d, extra);
    *dev_bytes = L.total;
    *host_bytes = (size_t)cfg->host_blocks * cfg->num_mla_layers * cfg->page_tokens * d.R;
    return HS_OK;
}

hs_status hs_pool_create(const hs_pool_config *cfg, void *dev_arena, size_t dev_bytes,
                         void *host_arena, size_t host_bytes, hs_pool **out) {
    if (!out) return HS_ERR_INVALID_ARG;
    *out = nullptr;
    size_t need_dev = 0, need_host = 0;
    hs_status st = hs_pool_required_bytes(cfg, &need_dev, &need_host);
    if (st != HS_OK) return st;
    if (!dev_arena || ((uintptr_t)dev_arena & 15)) return HS_ERR_INVALID_ARG;
    if (dev_bytes < need_dev || host_bytes < need_host) return HS_ERR_ARENA_TOO_SMALL;
    if (cfg->host_blocks > 0 && !host_arena) return HS_ERR_INVALID_ARG;

    hs_pool *p = new (std::nothrow) hs_pool();
    if (!p) return HS_ERR_INVALID_ARG;
    p->cfg = *cfg;
    Derived d = derive(cfg);
    p->R = d.R;
    p->nq_max = d.nq;
    p->C = d.C;
    p->hot_pages = d.hot_pages;
    p->max_pages = d.max_pages;
    p->idx_esize = d.esize;
    p->score_stride = d.score_stride;
    p->topk_nchunks = d.nchunks;
    p->attn_part_floats = d.attn_part_floats;
    size_t extra[16];
    p->layout = carve(cfg, d, extra);
    p->dev_base = (uint8_t *)dev_arena;
    p->host_base = (uint8_t *)host_arena;
    p->host_dev = nullptr;
    if (cfg->host_blocks > 0) {
        void *dp = nullptr;
        if (cudaHostGetDevicePointer(&dp, host_arena, 0) != cudaSuccess || !dp) {
            cudaGetLastError();
            delete p;
            return HS_ERR_INVALID_ARG;  // not pinned / not reachable from the device
        }
        p->host_dev = (uint8_t *)dp;
    }
    uint8_t *b = p->dev_base;
    const hs_layout &L = p->layout;
    p->d.rows = b + L.rows;
    p->d.idx_keys = b + L.idx_keys;
    p->d.idx_scale = (float *)(b + L.idx_scale);
    p->d.block_table = (int32_t *)(b + L.block_table);
    p->d.host_block_table = (int32_t *)(b + L.host_block_table);
    p->d.hot_map = (int32_t *)(b + L.hot_map);
    p->d.slot_token = (int32_t *)(b + L.slot_token);
    p->d.stamp = (uint32_t *)(b + L.stamp);
    p->d.hot_blocks = (int32_t *)(b + L.hot_blocks);
    p->d.seq_len = (int32_t *)(b + L.seq_len);
    p->d.req_step = (uint32_t *)(b + L.req_step);
    p->d.err = (int32_t *)(b + extra[0]);
    p->d.stats = (unsigned long long *)(b + extra[1]);
    p->d.scores = (float *)(b + extra[2]);
    p->d.topk_state = (hs::TopkRowState *)(b + extra[3]);
    p->d.topk_hist = (uint32_t *)(b + extra[4]);
    p->d.topk_chunk = (int32_t *)(b + extra[5]);
    p->d.miss_count = (int32_t *)(b + extra[6]);
    p->d.miss_tok = (int32_t *)(b + extra[7]);
    p->d.miss_slot = (int32_t *)(b + extra[8]);
    p->d.attn_part = (float *)(b + extra[9]);
    p->d.topk_cand = cfg->top_k <= hs::kTopkSampledMaxK ? (uint2 *)(b + extra[10]) : nullptr;

    p->has_key_map = false;
    if (cfg->idx_fmt == HS_IDX_E4M3 && cfg->idx_dim == 128) {
        if (!make_key_map(p)) {
            delete p;
            return HS_ERR_CUDA;
        }
        p->has_key_map = true;
    }
    const size_t maxR = cfg->max_requests;
    p->seq_len.assign(maxR, 0);
    p->mode.assign(maxR, -1);
    p->block_table.assign(maxR * p->max_pages, -1);
    p->host_block_table.assign(maxR * p->max_pages, -1);
    p->hot_blocks.assign(maxR * p->hot_pages, -1);
    p->host_ok.assign(maxR * p->max_pages, 0);
    p->precopy_pending = false;
    p->precopy_ev = nullptr;
    p->copy_stream = nullptr;
    p->copy_priority = 0;
    p->ev_plan = nullptr;
    p->free_gpu.resize(cfg->gpu_blocks);
    for (int64_t i = 0; i < cfg->gpu_blocks; i++) p->free_gpu[i] = (int32_t)(cfg->gpu_blocks - 1 - i);
    p->free_host.resize(cfg->host_blocks);
    for (int64_t i = 0; i < cfg->host_blocks; i++) p->free_host[i] = (int32_t)(cfg->host_blocks - 1 - i);

    // tables: -1 everywhere, counters and state 0
    cudaError_t e = cudaSuccess;
    auto ms = [&](void *ptr, int v, size_t n) {
        if (e == cudaSuccess) e = cudaMemset(ptr, v, n);
    };
    ms(p->d.block_table, 0xFF, maxR * p->max_pages * 4);
    ms(p->d.host_block_table, 0xFF, maxR * p->max_pages * 4);
    ms(p->d.hot_map, 0xFF, maxR * (size_t)cfg->max_tokens * 4);
    ms(p->d.slot_token, 0xFF, maxR * (size_t)p->C * 4);
    ms(p->d.stamp, 0, maxR * (size_t)p->C * 4);
    ms(p->d.hot_blocks, 0xFF, maxR * (size_t)p->hot_pages * 4);
    ms(p->d.seq_len, 0, maxR * 4);
    ms(p->d.req_step, 0, maxR * 4);
    ms(p->d.err, 0, 16);
    ms(p->d.stats, 0, 32);
    ms(p->d.miss_count, 0, maxR * 4);
    if (e == cudaSuccess) e = hs::setup_kernel_attributes(p);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->precopy_ev, cudaEventDisableTiming);
    if (e == cudaSuccess && cfg->host_blocks > 0) {
        int lo = 0, hi = 0;  // numerically lower = higher priority
        e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
        p->copy_priority = hi;
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&p->copy_stream, cudaStreamNonBlocking, hi);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_plan, cudaEventDisableTiming);
        p->ev_copy.assign(cfg->num_mla_layers, nullptr);
        p->tc_begin.assign(cfg->num_mla_layers, nullptr);
        p->tc_end.assign(cfg->num_mla_layers, nullptr);
        for (int l = 0; l < cfg->num_mla_layers && e == cudaSuccess; l++) {
            e = cudaEventCreateWithFlags(&p->ev_copy[l], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreate(&p->tc_begin[l]);
            if (e == cudaSuccess) e = cudaEventCreate(&p->tc_end[l]);
        }
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        hs_pool_destroy(p);
        return HS_ERR_CUDA;
    }
    *out = p;
    return HS_OK;
}

void hs_pool_destroy(hs_pool *pool) {
    if (!pool) return;
    if (pool->precopy_ev) {
        if (pool->precopy_pending) cudaEventSynchronize(pool->precopy_ev);  // copies into the host arena
        cudaEventDestroy(pool->precopy_ev);
    }
    if (pool->copy_stream) {
        cudaStreamSynchronize(pool->copy_stream);
        cudaStreamDestroy(pool->copy_stream);
    }
    if (pool->ev_plan) cudaEventDestroy(pool->ev_plan);
    for (cudaEvent_t ev : pool->ev_copy)
        if (ev) cudaEventDestroy(ev);
    for (cudaEvent_t ev : pool->tc_begin)
        if (ev) cudaEventDestroy(ev);
    for (cudaEvent_t ev : pool->tc_end)
        if (ev) cudaEventDestroy(ev);
    delete pool;
}

hs_status hs_pool_get_layout(const hs_pool *pool, hs_layout *out) {
    if (!pool || !out) return HS_ERR_INVALID_ARG;
    *out = pool->layout;
    return HS_OK;
}

int64_t hs_pool_free_gpu_blocks(const hs_pool *pool) {
    return pool ? (int64_t)pool->free_gpu.size() : -1;
}

hs_status hs_request_open(hs_pool *p, int32_t req, hs_mode mode) {
    if (!req_ok(p, req) || p->mode[req] != -1) return HS_ERR_INVALID_ARG;
    if (mode != HS_FULL && mode != HS_MIXED && mode != HS_ZERO) return HS_ERR_INVALID_ARG;
    if (mode != HS_FULL && p->cfg.host_blocks == 0) return HS_ERR_INVALID_ARG;
    cudaStream_t st = 0;
    if (mode != HS_FULL) {
        if ((int)p->free_gpu.size() < p->hot_pages) return HS_ERR_CAPACITY;
        for (int i = 0; i < p->hot_pages; i++) {
            p->hot_blocks[(size_t)req * p->hot_pages + i] = p->free_gpu.back();
            p->free_gpu.pop_back();
        }
    }
    p->mode[req] = mode;
    p->seq_len[req] = 0;
    cudaError_t e = reset_hot(p, req, st);
    if (e == cudaSuccess) e = upload_tables(p, req, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return cuda_status(e);
}

hs_status hs_append(hs_pool *p, int32_t req, const void *mla_rows, const void *idx_keys,
                    const float *idx_scale, int32_t n, cudaStream_t st) {
    if (!req_ok(p, req) || p->mode[req] < 0 || n < 0 || (n > 0 && (!mla_rows || !idx_keys)))
        return HS_ERR_INVALID_ARG;
    const int64_t N0 = p->seq_len[req], N1 = N0 + n;
    if (N1 > p->cfg.max_tokens) return HS_ERR_INVALID_ARG;
    if (n == 0) return HS_OK;
    const int P = p->cfg.page_tokens, L = p->cfg.num_mla_layers, R = p->R;
    const int mode = p->mode[req];
    const size_t mp = p->max_pages;
    int32_t *bt = p->block_table.data() + req * mp;
    int32_t *hbt = p->host_block_table.data() + req * mp;
    const int p0 = (int)(N0 / P), p1 = (int)((N1 - 1) / P);
    const int tail0 = first_tail_page(p, mode, N1);
    const bool has_host = p->cfg.host_blocks > 0;
    // capacity check before touching anything
    int need_gpu = 0, need_host = 0;
    for (int pg = p0; pg <= p1; pg++) {
        if (pg >= tail0 && bt[pg] < 0) need_gpu++;
        if (has_host && hbt[pg] < 0) need_host++;
    }
    int released = 0;
    if (mode == HS_MIXED)
        for (int pg = 0; pg < std::min(tail0, p0 + 1); pg++)
            if (bt[pg] >= 0) released++;
    if (need_gpu > (int)p->free_gpu.size() + released) return HS_ERR_CAPACITY;
    if (need_host > (int)p->free_host.size()) return HS_ERR_HOST_POOL_FULL;
    for (int pg = p0; pg <= p1; pg++) {
        if (has_host && hbt[pg] < 0) {
            hbt[pg] = p->free_host.back();
            p->free_host.pop_back();
        }
    }
    cudaError_t e = cudaSuccess;
    // pages that left the tail window (mixed mode): host copy first (the
    // page's earlier rows may live on the GPU only), then the block goes back
    if (mode == HS_MIXED) {
        std::vector<int> leaving;
        for (int pg = 0; pg < std::min(tail0, p0 + 1); pg++)
            if (bt[pg] >= 0) leaving.push_back(pg);
        e = secure_host_copies(p, req, leaving, st);
        for (int pg : leaving) {
            p->free_gpu.push_back(bt[pg]);
            bt[pg] = -1;
        }
    }
    for (int pg = p0; pg <= p1; pg++)
        if (pg >= tail0 && bt[pg] < 0) {
            bt[pg] = p->free_gpu.back();
            p->free_gpu.pop_back();
        }
    // rows of a resident page go to the GPU only (its host copy is left to
    // hs_precopy, or made when the page leaves); the others to the host pool
    uint8_t *ok = p->host_ok.data() + req * mp;
    const uint8_t *src = (const uint8_t *)mla_rows;
    for (int pg = p0; pg <= p1 && e == cudaSuccess; pg++) {
        const int64_t t0 = std::max<int64_t>(N0, (int64_t)pg * P);
        const int64_t t1 = std::min<int64_t>(N1, (int64_t)(pg + 1) * P);
        const size_t cnt = (size_t)(t1 - t0);
        const bool on_gpu = bt[pg] >= 0;
        uint8_t *base = on_gpu ? p->d.rows + (size_t)bt[pg] * block_bytes(p)
                               : p->host_base + (size_t)hbt[pg] * block_bytes(p);
        for (int l = 0; l < L && e == cudaSuccess; l++) {
            const uint8_t *s = src + ((size_t)(t0 - N0) * L + l) * R;
            uint8_t *dst = base + ((size_t)l * P + (t0 % P)) * R;
            e = cudaMemcpy2DAsync(dst, R, s, (size_t)L * R, R, cnt, cudaMemcpyDefault, st);
        }
        ok[pg] = on_gpu ? 0 : 1;
    }
    const size_t krow = (size_t)p->cfg.idx_dim * p->idx_esize;
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(p->d.idx_keys + ((size_t)req * p->cfg.max_tokens + N0) * krow, idx_keys,
                            (size_t)n * krow, cudaMemcpyDefault, st);
    std::vector<float> ones;
    if (e == cudaSuccess) {
        const float *sc = idx_scale;
        if (!sc) {
            ones.assign(n, 1.0f);
            sc = ones.data();
        }
        e = cudaMemcpyAsync(p->d.idx_scale + (size_t)req * p->cfg.max_tokens + N0, sc,
                            (size_t)n * 4, cudaMemcpyDefault, st);
    }
    p->seq_len[req] = (int32_t)N1;
    if (e == cudaSuccess) e = upload_tables(p, req, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return cuda_status(e);
}

static hs_status set_mode(hs_pool *p, int32_t req, int mode, cudaStream_t st) {
    if (!req_ok(p, req) || p->mode[req] < 0) return HS_ERR_INVALID_ARG;
    if (mode != HS_FULL && mode != HS_MIXED && mode != HS_ZERO) return HS_ERR_INVALID_ARG;
    const int cur = p->mode[req];
    if (cur == mode) return HS_OK;
    if (p->cfg.host_blocks == 0) return HS_ERR_INVALID_ARG;  // a flip needs the host copies
    const size_t mp = p->max_pages;
    int32_t *bt = p->block_table.data() + req * mp;
    int32_t *hbt = p->host_block_table.data() + req * mp;
    int32_t *hot = p->hot_blocks.data() + (size_t)req * p->hot_pages;
    const int P = p->cfg.page_tokens;
    const int64_t N = p->seq_len[req];
    const int npages = (int)((N + P - 1) / P);
    const int tail0 = first_tail_page(p, mode, N);  // pages >= tail0 are resident afterwards
    // check everything before touching anything
    int leave = 0, join = 0;
    for (int pg = 0; pg < npages; pg++) {
        if (hbt[pg] < 0) return HS_ERR_INVALID_ARG;  // every page has its host copy
        if (pg < tail0 && bt[pg] >= 0) leave++;
        if (pg >= tail0 && bt[pg] < 0) join++;
    }
    const int hot_in = (cur == HS_FULL) ? p->hot_pages : 0;   // a hot buffer to lease
    const int hot_out = (mode == HS_FULL) ? p->hot_pages : 0;  // a hot buffer to return
    if ((int64_t)p->free_gpu.size() + leave + hot_out < (int64_t)join + hot_in) return HS_ERR_CAPACITY;
    // pages leaving the GPU: their host copies first, then their blocks
    std::vector<int> leaving;
    for (int pg = 0; pg < npages; pg++)
        if (pg < tail0 && bt[pg] >= 0) leaving.push_back(pg);
    cudaError_t e = secure_host_copies(p, req, leaving, st);
    for (int pg : leaving) {
        p->free_gpu.push_back(bt[pg]);
        bt[pg] = -1;
    }
    if (hot_out)
        for (int i = 0; i < p->hot_pages; i++) {
            p->free_gpu.push_back(hot[i]);
            hot[i] = -1;
        }
    const size_t bb = block_bytes(p);
    for (int pg = tail0; pg < npages && e == cudaSuccess; pg++)
        if (bt[pg] < 0) {  // back onto the GPU: one block copied from the host pool
            bt[pg] = p->free_gpu.back();
            p->free_gpu.pop_back();
            e = cudaMemcpyAsync(p->d.rows + (size_t)bt[pg] * bb, p->host_base + (size_t)hbt[pg] * bb,
                                bb, cudaMemcpyHostToDevice, st);
        }
    if (hot_in)
        for (int i = 0; i < p->hot_pages; i++) {
            hot[i] = p->free_gpu.back();
            p->free_gpu.pop_back();
        }
    p->mode[req] = mode;
    if (e == cudaSuccess) e = reset_hot(p, req, st);
    if (e == cudaSuccess) e = upload_tables(p, req, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return cuda_status(e);
}

hs_status hs_request_set_mode(hs_pool *p, int32_t req, hs_mode mode, cudaStream_t st) {
    hs_status s = set_mode(p, req, mode, st);
    if (s == HS_OK) forget_policy(p, req);  // the caller now decides this request's residency
    return s;
}

hs_status hs_request_close(hs_pool *p, int32_t req) {
    if (!req_ok(p, req) || p->mode[req] < 0) return HS_ERR_INVALID_ARG;
    const size_t mp = p->max_pages;
    // a pre-copy may still read this request's blocks or write its host blocks
    if (p->precopy_pending && cudaEventSynchronize(p->precopy_ev) != cudaSuccess) return HS_ERR_CUDA;
    p->precopy_pending = false;
    std::fill(p->host_ok.begin() + req * mp, p->host_ok.begin() + (req + 1) * mp, 0);
    forget_policy(p, req);
    for (size_t pg = 0; pg < mp; pg++) {
        int32_t &g = p->block_table[req * mp + pg];
        if (g >= 0) p->free_gpu.push_back(g);
        g = -1;
        int32_t &h = p->host_block_table[req * mp + pg];
        if (h >= 0) p->free_host.push_back(h);
        h = -1;
    }
    for (int i = 0; i < p->hot_pages; i++) {
        int32_t &g = p->hot_blocks[(size_t)req * p->hot_pages + i];
        if (g >= 0) p->free_gpu.push_back(g);
        g = -1;
    }
    p->mode[req] = -1;
    p->seq_len[req] = 0;
    cudaError_t e = reset_hot(p, req, 0);
    if (e == cudaSuccess) e = upload_tables(p, req, 0);
    if (e == cudaSuccess) e = cudaStreamSynchronize(0);
    return cuda_status(e);
}

hs_status hs_precopy(hs_pool *p, cudaStream_t st, int64_t *pages) {
    if (pages) *pages = 0;
    if (!p || p->cfg.host_blocks == 0) return HS_ERR_INVALID_ARG;
    const int P = p->cfg.page_tokens;
    const size_t mp = p->max_pages;
    std::vector<std::pair<int32_t, int32_t>> pairs;
    std::vector<size_t> marked;
    for (int32_t r = 0; r < p->cfg.max_requests; r++) {
        if (p->mode[r] < 0) continue;
        const int complete = (int)(p->seq_len[r] / P);
        for (int pg = 0; pg < complete; pg++) {
            const size_t i = r * mp + pg;
            if (p->block_table[i] >= 0 && !p->host_ok[i] && p->host_block_table[i] >= 0) {
                pairs.push_back({p->block_table[i], p->host_block_table[i]});
                marked.push_back(i);
            }
        }
    }
    if (pairs.empty()) return HS_OK;
    // one event then covers every batch so far, whichever stream each used
    cudaError_t e = p->precopy_pending ? cudaStreamWaitEvent(st, p->precopy_ev, 0) : cudaSuccess;
    if (e == cudaSuccess) e = copy_blocks_to_host(p, pairs, st);
    if (e == cudaSuccess) e = cudaEventRecord(p->precopy_ev, st);
    if (e != cudaSuccess) return HS_ERR_CUDA;
    p->precopy_pending = true;
    for (size_t i : marked) p->host_ok[i] = 1;
    if (pages) *pages = (int64_t)pairs.size();
    return HS_OK;
}

hs_status hs_append_pressure(hs_pool *p, int32_t req, const void *mla_rows, const void *idx_keys,
                             const float *idx_scale, int32_t n, cudaStream_t st, int32_t *flipped,
                             int32_t *n_flipped) {
    if (n_flipped) *n_flipped = 0;
    if (!req_ok(p, req) || p->mode[req] < 0) return HS_ERR_INVALID_ARG;
    int nf = 0;
    for (;;) {
        hs_status s = hs_append(p, req, mla_rows, idx_keys, idx_scale, n, st);
        if (s != HS_ERR_CAPACITY || p->cfg.host_blocks == 0) return s;
        // the full-residency request with the most resident pages whose flip
        // frees blocks, lower id on ties
        int32_t x = -1;
        int best = -1;
        for (int32_t r = 0; r < p->cfg.max_requests; r++) {
            if (p->mode[r] != HS_FULL) continue;
            if (blocks_in_mode(p, r, HS_MIXED) >= blocks_in_mode(p, r, HS_FULL)) continue;
            const int res = resident_pages(p, r);
            if (res > best) {
                best = res;
                x = r;
            }
        }
        if (x < 0) return HS_ERR_CAPACITY;
        s = set_mode(p, x, HS_MIXED, st);
        if (s != HS_OK) return s;
        p->policy_flipped.push_back(x);
        if (flipped) flipped[nf] = x;
        nf++;
        if (n_flipped) *n_flipped = nf;
    }
}

hs_status hs_pool_relieve(hs_pool *p, cudaStream_t st, int32_t *restored, int32_t *n_restored) {
    if (n_restored) *n_restored = 0;
    if (!p) return HS_ERR_INVALID_ARG;
    int64_t open = 0;
    for (int32_t r = 0; r < p->cfg.max_requests; r++) open += p->mode[r] >= 0;
    int nr = 0;
    while (!p->policy_flipped.empty()) {
        const int32_t x = p->policy_flipped.back();
        // net blocks the return takes: every page back, the hot buffer given up
        const int64_t need = blocks_in_mode(p, x, HS_FULL) - blocks_in_mode(p, x, p->mode[x]);
        if ((int64_t)p->free_gpu.size() < need + open) break;  // keep one page per request free
        hs_status s = set_mode(p, x, HS_FULL, st);
        if (s != HS_OK) return s;
        p->policy_flipped.pop_back();
        if (restored) restored[nr] = x;
        nr++;
        if (n_restored) *n_restored = nr;
    }
    return HS_OK;
}

static bool aligned16(const void *ptr) { return ((uintptr_t)ptr & 15) == 0; }

static bool batch_ok(const hs_pool *p, int32_t B, int32_t nq) {
    if (!p || B <= 0 || B > p->cfg.max_requests || nq <= 0 || nq > p->nq_max) return false;
    for (int b = 0; b < B; b++)
        if (p->mode[b] < 0) return false;
    return true;
}

// Calls that score, select or resolve a request's tokens also need the cache
// to hold the step's own nq tokens (N >= nq; an empty request is refused).
static bool step_batch_ok(const hs_pool *p, int32_t B, int32_t nq) {
    if (!batch_ok(p, B, nq)) return false;
    for (int b = 0; b < B; b++)
        if (p->seq_len[b] < nq) return false;
    return true;
}

hs_status hs_indexer_score(hs_pool *p, const void *q, const float *w, int32_t B, int32_t nq,
                           float *scores, int64_t stride, cudaStream_t st) {
    if (!step_batch_ok(p, B, nq) || !q || !w || !scores || stride < p->cfg.max_tokens)
        return HS_ERR_INVALID_ARG;
    return cuda_status(hs::launch_indexer_score(p, q, w, B, nq, scores, stride, st));
}

hs_status hs_topk(hs_pool *p, const float *scores, int64_t stride, int32_t B, int32_t nq,
                  int32_t *topk, cudaStream_t st) {
    if (!step_batch_ok(p, B, nq) || !scores || !topk || stride < p->cfg.max_tokens)
        return HS_ERR_INVALID_ARG;
    return cuda_status(hs::launch_topk(p, scores, stride, B, nq, topk, st));
}

hs_status hs_indexer_topk(hs_pool *p, const void *q, const float *w, int32_t B, int32_t nq,
                          int32_t *topk, cudaStream_t st) {
    if (!step_batch_ok(p, B, nq) || !q || !w || !topk) return HS_ERR_INVALID_ARG;
    cudaError_t e = hs::launch_indexer_score(p, q, w, B, nq, p->d.scores, p->score_stride, st);
    if (e == cudaSuccess) e = hs::launch_topk(p, p->d.scores, p->score_stride, B, nq, topk, st);
    return cuda_status(e);
}

hs_status hs_resolve(hs_pool *p, const int32_t *topk, int32_t B, int32_t nq, int32_t *row_id,
                     cudaStream_t st) {
    if (!step_batch_ok(p, B, nq) || !topk || !row_id) return HS_ERR_INVALID_ARG;
    return cuda_status(hs::launch_resolve(p, topk, B, nq, row_id, st));
}

hs_status hs_resolve_plan(hs_pool *p, const int32_t *topk, int32_t B, int32_t nq, int32_t *row_id,
                          cudaStream_t st) {
    if (!step_batch_ok(p, B, nq) || !topk || !row_id) return HS_ERR_INVALID_ARG;
    return cuda_status(hs::launch_resolve_plan(p, topk, B, nq, row_id, st));
}

hs_status hs_miss_copy(hs_pool *p, int32_t B, int32_t nq, cudaStream_t st) {
    if (!step_batch_ok(p, B, nq)) return HS_ERR_INVALID_ARG;
    return cuda_status(hs::launch_miss_copy(p, B, nq, st));
}

hs_status hs_pool_time_copies(hs_pool *p, int32_t enable) {
    if (!p || p->cfg.host_blocks == 0) return HS_ERR_INVALID_ARG;
    p->time_copies = enable != 0;
    return HS_OK;
}

hs_status hs_pool_copy_times(hs_pool *p, float *ms, int32_t n) {
    if (!p || !ms || p->cfg.host_blocks == 0 || n < 0 || n > p->cfg.num_mla_layers)
        return HS_ERR_INVALID_ARG;
    for (int l = 0; l < n; l++) {
        const cudaError_t e = cudaEventElapsedTime(&ms[l], p->tc_begin[l], p->tc_end[l]);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return HS_ERR_CUDA;
        }
    }
    return HS_OK;
}

hs_status hs_miss_copy_layers(hs_pool *p, int32_t B, int32_t nq, int32_t l0, int32_t l1,
                              int32_t ctas, cudaStream_t st) {
    if (!step_batch_ok(p, B, nq) || l0 < 0 || l1 <= l0 || l1 > p->cfg.num_mla_layers || ctas < 0)
        return HS_ERR_INVALID_ARG;
    return cuda_status(hs::launch_miss_copy(p, B, nq, st, l0, l1, ctas));
}

hs_status hs_sparse_mla_decode(hs_pool *p, int32_t layer, const void *q, const int32_t *row_id,
                               int32_t B, int32_t nq, float scale, void *out, float *lse,
                               cudaStream_t st) {
    if (!batch_ok(p, B, nq) || !q || !row_id || !out || layer < 0 ||
        layer >= p->cfg.num_mla_layers || !aligned16(q) || !aligned16(out))
        return HS_ERR_INVALID_ARG;
    return cuda_status(hs::launch_attention(p, layer, q, row_id, B, nq, scale, out, lse, st));
}

// Resolve, then the attention of every layer.  Without a host pool there is
// nothing to copy: the plan and the attentions run on `st`.  With one, layer
// l's missed rows are copied on the pool's side stream (about 64 CTAs at a
// high launch priority) while layer l-1 attends on `st`: `st` waits for
// layer l's copy, by an event, just before layer l's attention.  (Copying the
// layers beside the attention with a full-width copy grid was measured
// slower at the mixed-residency MTP3 workload, 5.4-5.7 against 5.0 ms per
// step: both kernels' CTAs then shared every SM.)
// CTAs of a layer's copy that runs beside the attention: the link's rate
// with about 64 SMs (measured 189 GB/s against 192 for the full-width copy at
// the MTP3 workload), the other SMs left to the attention.
constexpr int kCopyCtasBeside = 64;

static cudaError_t resolve_attend(hs_pool *p, const int32_t *topk, int B, int nq,
                                  const void *q_mla, float scale, void *out, float *lse,
                                  int32_t *row_id, cudaStream_t st, bool q_ready) {
    const int H = p->cfg.mla_heads, L = p->cfg.num_mla_layers;
    const size_t qstride = (size_t)B * nq * H * hs::kLatent * 2;
    const size_t ostride = (size_t)B * nq * H * hs::kNope * 2;
    // beside the copies, an attention launches only once its layer's copy and
    // the previous layer are done (no early launch: its CTAs would hold SMs
    // the copy needs while they wait)
    const bool pdl = p->cfg.host_blocks == 0;
    auto attend = [&](int l) {
        return hs::launch_attention(p, l, (const uint8_t *)q_mla + l * qstride, row_id, B, nq, scale,
                                    (uint8_t *)out + l * ostride,
                                    lse ? lse + (size_t)l * B * nq * H : nullptr, st, q_ready, pdl);
    };
    if (p->cfg.host_blocks == 0) {
        cudaError_t e = hs::launch_resolve(p, topk, B, nq, row_id, st);
        for (int l = 0; l < L && e == cudaSuccess; l++) e = attend(l);
        return e;
    }
    cudaError_t e = hs::launch_resolve_plan(p, topk, B, nq, row_id, st);
    if (e == cudaSuccess) e = cudaEventRecord(p->ev_plan, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->copy_stream, p->ev_plan, 0);
    // timing records: external ones while the stream is being captured, so
    // that the graph records them at every replay; plain ones otherwise
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (e == cudaSuccess && p->time_copies) e = cudaStreamIsCapturing(p->copy_stream, &cap);
    auto stamp = [&](cudaEvent_t ev) {
        return cap == cudaStreamCaptureStatusActive
                   ? cudaEventRecordWithFlags(ev, p->copy_stream, cudaEventRecordExternal)
                   : cudaEventRecord(ev, p->copy_stream);
    };
    for (int l = 0; l < L && e == cudaSuccess; l++) {
        if (p->time_copies) e = stamp(p->tc_begin[l]);
        if (e == cudaSuccess)
            e = hs::launch_miss_copy(p, B, nq, p->copy_stream, l, l + 1, kCopyCtasBeside, p->copy_priority);
        if (e == cudaSuccess && p->time_copies) e = stamp(p->tc_end[l]);
        if (e == cudaSuccess) e = cudaEventRecord(p->ev_copy[l], p->copy_stream);
    }
    for (int l = 0; l < L && e == cudaSuccess; l++) {
        e = cudaStreamWaitEvent(st, p->ev_copy[l], 0);
        if (e == cudaSuccess) e = attend(l);
    }
    return e;
}

hs_status hs_resolve_attend(hs_pool *p, const int32_t *topk, int32_t B, int32_t nq,
                            const void *q_mla, float softmax_scale, void *out, float *lse,
                            int32_t *row_id, cudaStream_t st) {
    if (!step_batch_ok(p, B, nq) || !topk || !q_mla || !out || !row_id || !aligned16(q_mla) ||
        !aligned16(out))
        return HS_ERR_INVALID_ARG;
    return cuda_status(resolve_attend(p, topk, B, nq, q_mla, softmax_scale, out, lse, row_id, st,
                                      false));
}

hs_status hs_step(hs_pool *p, const hs_step_args *a, cudaStream_t st) {
    if (!a || !step_batch_ok(p, a->B, a->nq) || !a->q_idx || !a->w_idx || !a->q_mla || !a->out ||
        !a->topk || !a->row_id || !aligned16(a->q_mla) || !aligned16(a->out))
        return HS_ERR_INVALID_ARG;
    const int B = a->B, nq = a->nq;
    cudaError_t e = hs::launch_indexer_score(p, a->q_idx, a->w_idx, B, nq, p->d.scores,
                                             p->score_stride, st);
    if (e == cudaSuccess) e = hs::launch_topk(p, p->d.scores, p->score_stride, B, nq, a->topk, st);
    if (e == cudaSuccess)
        e = resolve_attend(p, a->topk_in ? a->topk_in : a->topk, B, nq, a->q_mla, a->softmax_scale,
                           a->out, a->lse, a->row_id, st, true);
    return cuda_status(e);
}

int32_t hs_step_kernel_count(const hs_pool *p, int32_t B, int32_t nq) {
    if (!p || B <= 0 || B > p->cfg.max_requests || nq <= 0 || nq > p->nq_max) return -1;
    // the step's resolve is the plan plus, with a host pool, one copy per layer
    const int L = p->cfg.num_mla_layers;
    return hs::indexer_kernel_count(p, B, nq) + hs::topk_kernel_count(p, B, nq) + 1 +
           (p->cfg.host_blocks > 0 ? L : 0) + L * hs::attention_kernel_count(p, B, nq);
}

hs_status hs_pool_get_error(hs_pool *p, hs_status *out) {
    if (!p || !out) return HS_ERR_INVALID_ARG;
    int32_t v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&v, p->d.err, 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(p->d.err, 0, 4);
    if (e != cudaSuccess) return HS_ERR_CUDA;
    *out = (hs_status)v;
    return HS_OK;
}

hs_status hs_pool_stats(hs_pool *p, hs_stats *out) {
    if (!p || !out) return HS_ERR_INVALID_ARG;
    unsigned long long v[4];
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(v, p->d.stats, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return HS_ERR_CUDA;
    out->resident = v[0];
    out->hits = v[1];
    out->misses = v[2];
    out->bytes_copied = v[3];
    return HS_OK;
}

hs_status hs_pool_reset_stats(hs_pool *p) {
    if (!p) return HS_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemset(p->d.stats, 0, 32);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    return cuda_status(e);
}

hs_status hs_pool_dump_state(hs_pool *p, int32_t req, int32_t *hot_map, int32_t *slot_token,
                             uint32_t *stamp, int32_t *block_table, int32_t *host_block_table,
                             int32_t *hot_blocks, uint32_t *step, int32_t *seq_len) {
    if (!req_ok(p, req)) return HS_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    const size_t maxT = p->cfg.max_tokens, C = p->C, mp = p->max_pages, hp = p->hot_pages;
    auto cp = [&](void *dst, const void *src, size_t n) {
        if (dst && e == cudaSuccess) e = cudaMemcpy(dst, src, n, cudaMemcpyDeviceToHost);
    };
    cp(hot_map, p->d.hot_map + req * maxT, maxT * 4);
    cp(slot_token, p->d.slot_token + req * C, C * 4);
    cp(stamp, p->d.stamp + req * C, C * 4);
    cp(block_table, p->d.block_table + req * mp, mp * 4);
    cp(host_block_table, p->d.host_block_table + req * mp, mp * 4);
    cp(hot_blocks, p->d.hot_blocks + req * hp, hp * 4);
    cp(step, p->d.req_step + req, 4);
    cp(seq_len, p->d.seq_len + req, 4);
    return cuda_status(e);
}

hs_status hs_pool_load_state(hs_pool *p, int32_t req, const int32_t *hot_map,
                             const int32_t *slot_token, const uint32_t *stamp, uint32_t step) {
    if (!req_ok(p, req) || p->mode[req] < 0 || !hot_map || !slot_token || !stamp)
        return HS_ERR_INVALID_ARG;
    const size_t maxT = p->cfg.max_tokens, C = p->C;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(p->d.hot_map + req * maxT, hot_map, maxT * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(p->d.slot_token + req * C, slot_token, C * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(p->d.stamp + req * C, stamp, C * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(p->d.req_step + req, &step, 4, cudaMemcpyHostToDevice);
    return cuda_status(e);
}

}  // extern "C"
