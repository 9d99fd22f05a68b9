// Private declarations shared by the translation units of libhs.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "hs.h"

namespace hs {

constexpr int kLatent = 576;
constexpr int kNope = 512;
constexpr int kRope = 64;
constexpr int kTopkChunk = 8192;   // scores per CTA in the top-K passes
constexpr int kTopkBins = 2048;    // 11-bit digit
constexpr int kTopkCandCap = 8192;    // candidates a row keeps in the sampled-threshold top-K
constexpr int kTopkSampledMaxK = 2048;  // largest K that path takes
constexpr int kMaxSplits = 32;     // split-K partials per attention query
constexpr int kNumSMs = 152;       // GB300

// Launch configuration with programmatic stream serialization (the kernel
// may start while the previous kernel on the stream finishes; it calls
// griddepcontrol.wait before its first global memory access) and, when
// cluster_z > 1, a (1, 1, cluster_z) or (cluster_x, 1, 1) cluster.
struct PdlLaunch {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attrs[3];  // room for one more attribute set by the caller
    PdlLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t st, dim3 cluster = dim3(1, 1, 1),
              bool pdl = true) {
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cfg.attrs = attrs;
        cfg.numAttrs = 0;
        if (pdl) {
            attrs[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attrs[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
            cfg.numAttrs++;
        }
        if (cluster.x * cluster.y * cluster.z > 1) {
            attrs[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
            attrs[cfg.numAttrs].val.clusterDim.x = cluster.x;
            attrs[cfg.numAttrs].val.clusterDim.y = cluster.y;
            attrs[cfg.numAttrs].val.clusterDim.z = cluster.z;
            cfg.numAttrs++;
        }
    }
};

// Per-row state of the radix top-K (one row = one (request, query)).
struct TopkRowState {
    uint32_t prefix;   // high digits of the threshold key found so far
    uint32_t mask;     // bits of `prefix` that are fixed
    int32_t need;      // rows still to take at/below the current prefix
    int32_t take_all;  // visible <= K: every visible token is selected
    uint32_t ticket;   // CTAs of this row done with the current pass
    int32_t visible;
    int32_t pad[2];
};

struct DevPtrs {
    uint8_t *rows;              // [gpu_blocks][L][P][R]
    uint8_t *idx_keys;          // [maxR][maxT][Di * esize]
    float *idx_scale;           // [maxR][maxT]
    int32_t *block_table;       // [maxR][maxPages]
    int32_t *host_block_table;  // [maxR][maxPages]
    int32_t *hot_map;           // [maxR][maxT]
    int32_t *slot_token;        // [maxR][C]
    uint32_t *stamp;            // [maxR][C]
    int32_t *hot_blocks;        // [maxR][C/P]
    int32_t *seq_len;           // [maxR]
    uint32_t *req_step;         // [maxR]
    int32_t *err;               // sticky error word
    unsigned long long *stats;  // resident, hits, misses, bytes
    float *scores;              // [maxR*nq][score_stride]
    TopkRowState *topk_state;   // [maxR*nq]
    uint32_t *topk_hist;        // [maxR*nq][kTopkBins]
    int32_t *topk_chunk;        // [maxR*nq][nchunks][2]
    uint2 *topk_cand;           // [maxR*nq][kTopkCandCap] (key, token); null when K > kTopkSampledMaxK
    int32_t *miss_count;        // [maxR]
    int32_t *miss_tok;          // [maxR][nq*K]
    int32_t *miss_slot;         // [maxR][nq*K]
    float *attn_part;           // split-K partials
};

}  // namespace hs

struct hs_pool {
    hs_pool_config cfg;
    int R;            // row bytes
    int nq_max;       // num_spec + 1
    int C;            // hot rows per request
    int hot_pages;    // C / P
    int max_pages;    // ceil(max_tokens / P)
    int idx_esize;    // 1 (E4M3) or 4 (fp32)
    int64_t score_stride;
    int topk_nchunks;
    size_t attn_part_floats;
    hs_layout layout;
    uint8_t *dev_base;
    uint8_t *host_base;      // host pointer of the pinned host pool
    uint8_t *host_dev;       // the same memory as seen from the device
    hs::DevPtrs d;
    CUtensorMap key_map;     // TMA map of the indexer key slab (E4M3, dim 128)
    bool has_key_map;
    // host mirrors
    std::vector<int32_t> seq_len;
    std::vector<int32_t> mode;  // -1 = closed
    std::vector<int32_t> block_table;
    std::vector<int32_t> host_block_table;
    std::vector<int32_t> hot_blocks;
    std::vector<int32_t> free_gpu;
    std::vector<int32_t> free_host;
    // host_ok[req * max_pages + page]: the pinned host pool holds every token
    // appended to the page so far (or a pre-copy of it is enqueued)
    std::vector<uint8_t> host_ok;
    cudaEvent_t precopy_ev;  // recorded after the last pre-copy batch
    bool precopy_pending;    // a pre-copy batch was enqueued and not waited for
    std::vector<int32_t> policy_flipped;  // requests the pressure policy flipped, in order
    // with a host pool: the side stream that copies a step's missed rows layer by
    // layer beside the attention, and the events that order the two
    cudaStream_t copy_stream;
    int copy_priority;
    cudaEvent_t ev_plan;
    std::vector<cudaEvent_t> ev_copy;  // [L]
    // timing of the side stream's per-layer copies (hs_pool_time_copies)
    bool time_copies;
    std::vector<cudaEvent_t> tc_begin, tc_end;  // [L]
};

namespace hs {

// Device-side error recording (first error wins, never traps).
__device__ __forceinline__ void set_error(int32_t *err, int code) {
    atomicCAS(err, 0, code);
}

// ---- launchers (each returns cudaGetLastError() after enqueueing) ----
cudaError_t launch_indexer_score(const hs_pool *p, const void *q, const float *w, int B, int nq,
                                 float *scores, int64_t stride, cudaStream_t st);
cudaError_t launch_topk(const hs_pool *p, const float *scores, int64_t stride, int B, int nq,
                        int32_t *topk, cudaStream_t st);
cudaError_t launch_resolve(const hs_pool *p, const int32_t *topk, int B, int nq, int32_t *row_id,
                           cudaStream_t st);
cudaError_t launch_resolve_plan(const hs_pool *p, const int32_t *topk, int B, int nq,
                                int32_t *row_id, cudaStream_t st);
// Miss rows of layers [l0, l1) (l1 < 0: through the last layer).
cudaError_t launch_miss_copy(const hs_pool *p, int B, int nq, cudaStream_t st, int l0 = 0,
                             int l1 = -1, int ctas = 0, int priority = 0);
// q_ready: the queries were written before the previous kernel on `st`
// started (true inside hs_step), so the kernel may stage them before it waits
// for that kernel.
cudaError_t launch_attention(const hs_pool *p, int layer, const void *q, const int32_t *row_id,
                             int B, int nq, float scale, void *out, float *lse, cudaStream_t st,
                             bool q_ready = false, bool pdl = true);
int indexer_kernel_count(const hs_pool *p, int B, int nq);
int topk_kernel_count(const hs_pool *p, int B, int nq);
int resolve_kernel_count(const hs_pool *p, int B, int nq);
int attention_kernel_count(const hs_pool *p, int B, int nq);
cudaError_t setup_kernel_attributes(const hs_pool *p);
size_t attention_partial_floats(const hs_pool_config *c);

}  // namespace hs
