/*
 * Plain CPU oracle for the Hybrid HiSparse sparse-MLA decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no source, header, table or helper with the
 * CUDA library; it is written to be read against the pages, not to be fast.
 *
 * Sources (web pages on vLLM's Hybrid HiSparse):
 *   [A] "Un contexte d'un million sur huit H200"
 *       - "Ce qui se passe": an indexer picks the top-K tokens and sparse MLA
 *         attends only to those; one indexer layer serves four sparse-MLA
 *         layers (IndexShare); the indexer cache stays resident.
 *       - "Les trois états de résidence": full / mixed / zero residency; in
 *         mixed residency the tail stays on the GPU and is never evicted,
 *         selected rows of older pages go to hot buffers; one fused resolve
 *         reads resident rows in place, refreshes the LRU entry of hot rows
 *         and copies exactly one row from pinned host memory on a miss.
 *       - "Ce qu'il faut en retenir": hot buffers hold 2*top-K rows, and
 *         (num_speculative_tokens+2)*top-K under MTP.
 *   [B] "vLLM sert GLM-5.3 en contexte 1M sur 16 H200"
 *       - "Comment s'y prendre": top-K is 2048 selected tokens; when the
 *         prompt fits inside those 2048 tokens the sparse kernel equals the
 *         dense path (the dense/sparse equivalence pinned by the tests).
 *
 * Everything the pages leave open is taken as stated beside each function
 * (the "reading").  Floating point is fp64 except where the method fixes the
 * stored type (indexer scores are stored as fp32; their inputs are built so
 * that every sum is exact, which makes the order of summation irrelevant).
 *
 * Parity status per function:
 *   hso_e4m3 ................ pinned (OCP FP8 E4M3FN table, torch decode)
 *   hso_dequant_row ......... pinned (hand-built rows with known values)
 *   hso_indexer_scores ...... pinned (int64 recomputation, exact)
 *   hso_topk ................ pinned (brute force, invariants)
 *   hso_resolve ............. pinned (history-replay LRU, invariants)
 *   hso_attention ........... pinned (K >= N equals dense SDPA in fp64,
 *                                     one-row and equal-score closed forms)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status codes, numbered like the library's so the tests can compare. */
enum { HSO_OK = 0, HSO_ERR_CAPACITY = 3, HSO_ERR_INDEX_RANGE = 5 };

/* Row storage formats of one MLA latent row (576 values: 512 "nope" + 64 rope). */
enum { HSO_ROW_E4M3_656 = 0, HSO_ROW_F32_2304 = 1 };
/* Indexer query/key element formats. */
enum { HSO_IDX_E4M3 = 0, HSO_IDX_F32 = 1 };

#define HSO_LATENT 576
#define HSO_NOPE 512

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* OCP 8-bit floating point, E4M3FN: 1 sign bit, 4 exponent bits (bias 7),
 * 3 mantissa bits, no infinities, S.1111.111 is NaN, exponent 0 is
 * subnormal (m/8 * 2^-6). */
double hso_e4m3(uint8_t b)
{
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double hso_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

int hso_row_bytes(int fmt)
{
    return fmt == HSO_ROW_E4M3_656 ? 656 : 2304;
}

/* One stored latent row -> 576 doubles.
 * Reading of the "FP8 KV cache" row (the pages name only FP8 latent rows):
 * bytes [0,512) are E4M3 codes of the 512 nope dims, bytes [512,528) four
 * fp32 scales, one per group of 128 nope dims, bytes [528,656) the 64 rope
 * dims in bf16.  The F32 format is 576 plain fp32 values. */
void hso_dequant_row(int fmt, const uint8_t *row, double *out)
{
    int i;
    if (fmt == HSO_ROW_E4M3_656) {
        float sc[4];
        memcpy(sc, row + 512, sizeof sc);
        for (i = 0; i < HSO_NOPE; i++)
            out[i] = hso_e4m3(row[i]) * (double)sc[i / 128];
        for (i = 0; i < 64; i++) {
            uint16_t h;
            memcpy(&h, row + 528 + 2 * i, 2);
            out[HSO_NOPE + i] = hso_bf16(h);
        }
    } else {
        for (i = 0; i < HSO_LATENT; i++) {
            float f;
            memcpy(&f, row + 4 * i, 4);
            out[i] = (double)f;
        }
    }
}

static double idx_elem(int fmt, const void *base, size_t i)
{
    if (fmt == HSO_IDX_E4M3)
        return hso_e4m3(((const uint8_t *)base)[i]);
    return (double)((const float *)base)[i];
}

/* ------------------------------------------------------------------------ */
/* Indexer score ("Ce qui se passe": the indexer scores every cached token)  */
/* ------------------------------------------------------------------------ */

/* Reading: the pages name an indexer with heads and nothing more.  We take
 * the lightning-indexer form
 *     s[j][t] = sum_h w[j][h] * ReLU(sigma[t] * (q[j][h][:] . k[t][:]))
 * with ReLU(x) = x if x > 0 else +0.  Compiling with -DHSO_IDENTITY_GATE
 * takes the identity gate instead (gate(x) = x), the other plain reading of
 * the unnamed indexer; hso_gate_is_identity() says which one was built.  Query j of the nq queries of a step
 * sees tokens t in [0, N - nq + j + 1) (its own position included); the other
 * entries are set to -inf.
 *   q: [nq][Hi][Di], w: [nq][Hi] fp32, keys: [N][Di], sigma: [N] fp32,
 *   s: [nq][N] fp32 (output). */
#ifdef HSO_IDENTITY_GATE
#define HSO_GATE(x) (x)
int hso_gate_is_identity(void) { return 1; }
#else
#define HSO_GATE(x) ((x) > 0.0 ? (x) : 0.0)
int hso_gate_is_identity(void) { return 0; }
#endif

void hso_indexer_scores(int idx_fmt, const void *q, const float *w,
                        const void *keys, const float *sigma,
                        int N, int nq, int Hi, int Di, float *s)
{
    int j;
    for (j = 0; j < nq; j++) {
        int visible = N - nq + j + 1;
        int t;
#pragma omp parallel for schedule(static)
        for (t = 0; t < N; t++) {
            double acc = 0.0;
            int h;
            if (t >= visible) {
                s[(size_t)j * N + t] = -INFINITY;
                continue;
            }
            for (h = 0; h < Hi; h++) {
                double dot = 0.0, x;
                int d;
                for (d = 0; d < Di; d++)
                    dot += idx_elem(idx_fmt, q, ((size_t)j * Hi + h) * Di + d) *
                           idx_elem(idx_fmt, keys, (size_t)t * Di + d);
                x = (double)sigma[t] * dot;
                acc += (double)w[j * Hi + h] * HSO_GATE(x);
            }
            s[(size_t)j * N + t] = (float)acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Top-K ("Comment s'y prendre": the 2048 selected tokens)                    */
/* ------------------------------------------------------------------------ */

typedef struct {
    float s;
    int32_t t;
} hso_pair;

static int cmp_desc_score(const void *a, const void *b)
{
    const hso_pair *x = (const hso_pair *)a, *y = (const hso_pair *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->t > y->t) - (x->t < y->t);
}

static int cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* The K highest scores among t in [0, visible); equal scores go to the
 * lower token index; the chosen indices are written in ascending order and
 * the rest of out[0..K) is -1.  K >= visible selects every visible token.
 * A full sort, as plain as it gets. */
void hso_topk(const float *s, int visible, int K, int32_t *out)
{
    hso_pair *p = (hso_pair *)malloc(sizeof(hso_pair) * (size_t)(visible > 0 ? visible : 1));
    int t, m;
    for (t = 0; t < visible; t++) {
        p[t].s = s[t];
        p[t].t = t;
    }
    qsort(p, (size_t)visible, sizeof(hso_pair), cmp_desc_score);
    m = visible < K ? visible : K;
    for (t = 0; t < m; t++)
        out[t] = p[t].t;
    qsort(out, (size_t)m, sizeof(int32_t), cmp_i32);
    for (t = m; t < K; t++)
        out[t] = -1;
    free(p);
}

/* ------------------------------------------------------------------------ */
/* Fused resolve ("Les trois états de résidence")                            */
/* ------------------------------------------------------------------------ */

typedef struct {
    uint32_t stamp;
    int32_t slot;
} hso_slotkey;

static int cmp_slotkey(const void *a, const void *b)
{
    const hso_slotkey *x = (const hso_slotkey *)a, *y = (const hso_slotkey *)b;
    if (x->stamp != y->stamp) return x->stamp < y->stamp ? -1 : 1;
    return (x->slot > y->slot) - (x->slot < y->slot);
}

/* One request, one decode step.
 *
 * State (per request, updated in place):
 *   hot_map[t]     hot-buffer slot holding token t, or -1       [max_tokens]
 *   slot_token[c]  token held by slot c, or -1                  [C]
 *   stamp[c]       step of the slot's last use, 0 = never       [C]
 *   *step          number of the last step resolved (steps count from 1)
 * page_resident[p] is 1 when page p (tokens [p*P, (p+1)*P)) has a GPU copy
 * that is read in place (a full-residency page or a page of the tail).
 *
 * Steps, in the order the section describes them, with our readings:
 *  1. The nq selected lists are merged into U, their sorted union without
 *     duplicates (one row is fetched once even if several MTP queries ask).
 *  2. Each u in U is, in this precedence: resident (its page is on the GPU;
 *     read in place), a hit (hot_map[u] >= 0; the LRU entry is refreshed:
 *     stamp = this step) or a miss.
 *  3. LRU eviction: the slots not used in this step (stamp < step) are
 *     ordered by (stamp, slot); the first M of them, M = number of misses,
 *     are the victims (never-used slots have stamp 0 and go first).  Fewer
 *     than M such slots (only possible with a hot buffer below nq*K rows) is
 *     a capacity error, handled gracefully: every such slot is a victim, the
 *     first of the misses in ascending token order take them, the others
 *     read nothing (located as 0, like padding), and the step still counts.
 *  4. The i-th miss in ascending token order goes to the i-th victim in
 *     ascending slot order (the pages do not say which victim takes which
 *     row; this is our canonical choice).  The evicted token leaves hot_map;
 *     the new token enters it with stamp = step.
 *  5. Each selected entry (j,k) is located: loc_kind 1 = resident, value =
 *     the token; 2 = hot buffer, value = the slot; 0 = padding (-1 entry).
 * Outputs: loc_kind/loc_val [nq][K]; the misses that got a slot, in order
 * (miss_tok, miss_slot, *n_miss); counts[0..3) = resident, hit, copied miss
 * over U.  Returns HSO_OK, HSO_ERR_INDEX_RANGE (an index outside [0,N);
 * nothing changes) or HSO_ERR_CAPACITY (fewer free-able slots than misses;
 * the step is carried out as described in 3). */
int hso_resolve(int32_t *hot_map, int32_t *slot_token, uint32_t *stamp,
                uint32_t *step_io, int C, const uint8_t *page_resident,
                int P, int N, const int32_t *idx, int nq, int K,
                int32_t *loc_kind, int32_t *loc_val, int32_t *miss_tok,
                int32_t *miss_slot, int32_t *n_miss, int32_t *counts)
{
    uint32_t step = *step_io + 1;
    int32_t *U = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nq * K + 1));
    int32_t *slot_of = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nq * K + 1));
    hso_slotkey *cand = (hso_slotkey *)malloc(sizeof(hso_slotkey) * (size_t)(C + 1));
    int32_t *victim = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nq * K + 1));
    int nu = 0, i, j, k, m = 0, nc = 0, status = HSO_OK;

    counts[0] = counts[1] = counts[2] = 0;
    *n_miss = 0;

    /* 1. union */
    for (j = 0; j < nq * K; j++)
        if (idx[j] >= 0)
            U[nu++] = idx[j];
        else if (idx[j] != -1)
            status = HSO_ERR_INDEX_RANGE;
    qsort(U, (size_t)nu, sizeof(int32_t), cmp_i32);
    {
        int w = 0;
        for (i = 0; i < nu; i++)
            if (i == 0 || U[i] != U[i - 1])
                U[w++] = U[i];
        nu = w;
    }
    for (i = 0; i < nu; i++)
        if (U[i] >= N)
            status = HSO_ERR_INDEX_RANGE;
    if (status != HSO_OK)
        goto done;

    /* 2. classify; hits refresh their stamp */
    for (i = 0; i < nu; i++) {
        int32_t u = U[i];
        if (page_resident[u / P]) {
            slot_of[i] = -1;
            counts[0]++;
        } else if (hot_map[u] >= 0) {
            slot_of[i] = hot_map[u];
            stamp[hot_map[u]] = step;
            counts[1]++;
        } else {
            slot_of[i] = -2; /* miss, slot assigned below */
            miss_tok[m++] = u;
        }
    }

    /* 3. victims: least recently used slots not touched in this step */
    for (i = 0; i < C; i++)
        if (stamp[i] < step) {
            cand[nc].stamp = stamp[i];
            cand[nc].slot = i;
            nc++;
        }
    if (nc < m) { /* capacity error: the first nc misses get the nc slots */
        status = HSO_ERR_CAPACITY;
        m = nc;
    }
    counts[2] = m;
    qsort(cand, (size_t)nc, sizeof(hso_slotkey), cmp_slotkey);
    for (i = 0; i < m; i++)
        victim[i] = cand[i].slot;
    qsort(victim, (size_t)m, sizeof(int32_t), cmp_i32);

    /* 4. assignment */
    for (i = 0; i < m; i++) {
        int32_t c = victim[i], u = miss_tok[i];
        if (slot_token[c] >= 0)
            hot_map[slot_token[c]] = -1;
        slot_token[c] = u;
        hot_map[u] = c;
        stamp[c] = step;
        miss_slot[i] = c;
    }
    *n_miss = m;
    for (i = 0, k = 0; i < nu; i++)
        if (slot_of[i] == -2)
            slot_of[i] = k < m ? victim[k++] : -3; /* -3: a miss left without a slot */

    /* 5. locations */
    for (j = 0; j < nq * K; j++) {
        int32_t u = idx[j];
        int lo = 0, hi = nu - 1;
        if (u < 0) {
            loc_kind[j] = 0;
            loc_val[j] = -1;
            continue;
        }
        while (lo < hi) { /* U is sorted and contains u */
            int mid = (lo + hi) / 2;
            if (U[mid] < u) lo = mid + 1; else hi = mid;
        }
        if (slot_of[lo] == -1) {
            loc_kind[j] = 1;
            loc_val[j] = u;
        } else if (slot_of[lo] == -3) {
            loc_kind[j] = 0;
            loc_val[j] = -1;
        } else {
            loc_kind[j] = 2;
            loc_val[j] = slot_of[lo];
        }
    }
    *step_io = step;
done:
    free(U);
    free(slot_of);
    free(cand);
    free(victim);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Sparse MLA attention ("Ce qui se passe": attention over the top-K only)  */
/* ------------------------------------------------------------------------ */

/* Absorbed-MLA decode for one query position, all heads (reading: the pages
 * give only "latent"; we use the standard absorbed form where the 576-dim
 * latent row is both key and, in its first 512 dims, value):
 *   z[h][r] = tau * sum_{i<576} q[h][i] * row_r[i]        for rows with mask
 *   p[h][.] = softmax over the masked-in rows (the others are -inf)
 *   o[h][i] = sum_r p[h][r] * row_r[i],  i < 512
 *   lse[h]  = log(sum_r exp(z[h][r]))  (natural log)
 * q is bf16 [H][576]; rows are n stored rows of format fmt; mask may be NULL
 * (all rows in).  With no row in, o = 0 and lse = -inf. */
void hso_attention(int fmt, const uint16_t *q, int H, const uint8_t *rows,
                   const uint8_t *mask, int n, double tau, double *o,
                   double *lse)
{
    int R = hso_row_bytes(fmt);
    double *kv = (double *)malloc(sizeof(double) * (size_t)HSO_LATENT * (size_t)(n > 0 ? n : 1));
    int r, h;
    for (r = 0; r < n; r++)
        hso_dequant_row(fmt, rows + (size_t)r * R, kv + (size_t)r * HSO_LATENT);
#pragma omp parallel for schedule(static)
    for (h = 0; h < H; h++) {
        double qh[HSO_LATENT];
        double *z = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        double mx = -INFINITY, l = 0.0;
        int i, rr;
        for (i = 0; i < HSO_LATENT; i++)
            qh[i] = hso_bf16(q[(size_t)h * HSO_LATENT + i]);
        for (rr = 0; rr < n; rr++) {
            double dot = 0.0;
            if (mask && !mask[rr]) {
                z[rr] = -INFINITY;
                continue;
            }
            for (i = 0; i < HSO_LATENT; i++)
                dot += qh[i] * kv[(size_t)rr * HSO_LATENT + i];
            z[rr] = tau * dot;
            if (z[rr] > mx) mx = z[rr];
        }
        for (i = 0; i < HSO_NOPE; i++)
            o[(size_t)h * HSO_NOPE + i] = 0.0;
        if (mx == -INFINITY) {
            lse[h] = -INFINITY;
            free(z);
            continue;
        }
        for (rr = 0; rr < n; rr++) {
            double p;
            if (z[rr] == -INFINITY) continue;
            p = exp(z[rr] - mx);
            l += p;
            for (i = 0; i < HSO_NOPE; i++)
                o[(size_t)h * HSO_NOPE + i] += p * kv[(size_t)rr * HSO_LATENT + i];
        }
        for (i = 0; i < HSO_NOPE; i++)
            o[(size_t)h * HSO_NOPE + i] /= l;
        lse[h] = mx + log(l);
        free(z);
    }
    free(kv);
}
