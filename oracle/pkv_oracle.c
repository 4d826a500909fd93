/*
 * CPU oracle for the block-paged KV attention path.  TEST INFRASTRUCTURE ONLY:
 * it is loaded by tests/, by the package's smoke check and by the CPU-baseline
 * leg of the benchmark, never by the library.  It shares no code, header or
 * table with the CUDA library.
 *
 * Plain loops, no blocking, no fusion.  Inputs are read exactly (float32, or
 * bf16 widened bit-for-bit, E4M3 codes decoded exactly) and every sum, max,
 * exp and division is carried out in IEEE double; the one float32 step is the
 * FP8 append's quotient x / scale, whose rounding decides the stored code.
 *
 * What it follows (page titles as printed at the top of each page):
 *   "paged-cache.md" (mlx-node): requests keep K/V in fixed-size blocks of a
 *     per-layer pool (LayerKVPool row of the type table), reached through a
 *     per-request block table; refcounted prefix blocks are shared; a sliding
 *     group keeps absolute logical positions and replaces expired blocks by a
 *     null sentinel (Gemma4 coordinator section).
 *   "perf.md" (mlx-node), paged knob table: the graph-native K/V write puts the
 *     new rows into their pool slots (MLX_PAGED_NATIVE_KV_WRITE), decode
 *     gathers the pages through the table and attends them
 *     (MLX_PAGED_GRAPH_DECODE_GATHER; a sliding group reads from its first live
 *     block), and a prefill chunk attends a paged cached prefix
 *     (gather_kv_for_prefill_chunk bridge).
 * The attention itself is scaled dot-product attention with a softmax over the
 * keys in range; its plain definition is what is written below.
 *
 * Readings where the pages are silent:
 *   - pool layout [block][kv_head][slot][dim]; slot = block * block_size + offset
 *     (the vLLM convention the pages say they follow); a negative slot is skipped;
 *   - query head h reads kv head h / (Hq / Hkv);
 *   - window W > 0: the query at absolute position p attends positions
 *     max(0, p - W + 1) .. p; W = 0 is full attention;
 *   - seq_lens count the tokens just appended; the decode query sits at L - 1;
 *   - an empty key range gives an all-zero output;
 *   - FP8 pools ("perf.md" quantisation table: the paged adapter keeps an FP8
 *     KV cache with per-layer scales): each K/V element is one E4M3 code c
 *     holding the value e4m3(c) * scale, with one float32 scale for the K
 *     pool and one for the V pool of the layer; the append stores
 *     c = nearest E4M3 code to the float32 quotient x / scale (ties to the
 *     even code, magnitudes past 448 saturate to +-448); queries and new rows
 *     are bf16.  An FP8 block holds 16 tokens and head_dim is a multiple of
 *     64; the bytes of a (block, kv head) tile follow the order given at
 *     fp8_k_byte / fp8_v_byte below (a storage format of this library).
 *
 * PLANT_* macros compile deliberate mistakes; the pin tests build those
 * variants to show that each mistake is caught.  The normal build defines none.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1
#define OR_FP8 2 /* E4M3 pools, bf16 queries and new rows */

static double ld(const void *base, int dtype, size_t i)
{
    if (dtype == OR_BF16) {
        uint32_t u = (uint32_t)((const uint16_t *)base)[i] << 16;
        float f;
        memcpy(&f, &u, 4);
        return (double)f;
    }
    return (double)((const float *)base)[i];
}

static size_t esize(int dtype) { return dtype == OR_BF16 ? 2 : 4; }

/* ---------------------------------------------------------------------------
 * E4M3 ("FP8 Formats for Deep Learning", Micikevicius et al. 2022, the E4M3
 * column of its format table): sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits.  Exponent field 0 holds the subnormals m * 2^-9; the code
 * S.1111.111 is NaN; there is no infinity, so the largest magnitude is
 * 1.75 * 2^8 = 448.
 * ------------------------------------------------------------------------- */
static double e4m3_value(uint8_t c)
{
    int e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return (c & 0x80) ? -v : v;
}

/* Nearest finite E4M3 code to x: a search of the positive codes, whose
 * values increase with the code; a tie between two neighbours goes to the
 * one with an even code (mantissa lsb 0).  448 is the nearest finite value to
 * anything larger, so the search itself saturates.  The sign bit is x's own
 * (so -0.0 and negative values that round to zero give 0x80).  NaN gives
 * 0x7F. */
static double e4m3_grid[0x7F]; /* values of the codes 0x00 .. 0x7E */
static int e4m3_grid_ready;

static uint8_t e4m3_encode(float x)
{
    if (isnan(x)) return 0x7F;
    if (!e4m3_grid_ready) {
        for (int c = 0; c <= 0x7E; ++c) e4m3_grid[c] = e4m3_value((uint8_t)c);
        e4m3_grid_ready = 1;
    }
    double a = fabs((double)x);
    /* lo = the largest code whose value is <= a (bisection on the grid) */
    int lo = 0, hi = 0x7E;
    if (a >= e4m3_grid[0x7E]) {
        lo = 0x7E;
    } else {
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (e4m3_grid[mid] <= a) lo = mid; else hi = mid;
        }
    }
    int best = lo;
    if (lo < 0x7E) {
        double dl = a - e4m3_grid[lo], dh = e4m3_grid[lo + 1] - a;
#ifdef PLANT_E4M3_TIES
        if (dh < dl) best = lo + 1; /* wrong: ties go to the smaller magnitude */
#else
        if (dh < dl || (dh == dl && ((lo + 1) & 1) == 0)) best = lo + 1;
#endif
    }
    return (uint8_t)(signbit(x) ? (best | 0x80) : best);
}

void or_e4m3_decode(const uint8_t *codes, int32_t n, double *out)
{
    for (int32_t i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
}

void or_e4m3_encode(const float *x, int32_t n, uint8_t *out)
{
    for (int32_t i = 0; i < n; ++i) out[i] = e4m3_encode(x[i]);
}

/* Byte of (token t, dim d) inside one (block, kv head) tile of an FP8 pool
 * (16 tokens, dim a multiple of 64).  The order is the operand order of the
 * m16n8k16 tensor-core product, so that each of 32 threads finds its operand
 * values as 16 consecutive bytes:
 *   K: per 64-dim group, two 512-byte halves (tokens 0-7, 8-15); inside a
 *      half, 16 bytes per (token t%8, pair class c) holding, for each of the
 *      four 16-dim steps kk, the dims kk*16 + {2c, 2c+1, 2c+8, 2c+9};
 *   V: per 32-dim group of 512 bytes, 16 bytes per (dim d%8, pair class c)
 *      holding, for each of the four 8-dim steps, that dim's tokens
 *      {2c, 2c+1, 2c+8, 2c+9}. */
static size_t fp8_k_byte(int32_t t, int32_t d)
{
    int32_t r = d % 64, kk = r / 16, kap = r % 16;
    int32_t c = (kap % 8) / 2, j = (kap % 2) + 2 * (kap / 8);
    return (size_t)(d / 64) * 1024 + (size_t)(t / 8) * 512 + (size_t)((t % 8) * 4 + c) * 16 +
           (size_t)(kk * 4 + j);
}

static size_t fp8_v_byte(int32_t t, int32_t d)
{
#ifdef PLANT_FP8_VPERM
    int32_t c = (t % 8) / 2, j = (t % 2) * 2 + (t / 8); /* wrong: token pair order swapped */
#else
    int32_t c = (t % 8) / 2, j = (t % 2) + 2 * (t / 8);
#endif
    return (size_t)(d / 32) * 512 + (size_t)((d % 8) * 4 + c) * 16 + (size_t)(((d % 32) / 8) * 4 + j);
}

/* Pool element (block b, kv head g, slot offset t, dim d). */
static size_t pool_index(int32_t hkv, int32_t bs, int32_t dim, int32_t b, int32_t g, int32_t t,
                         int32_t d)
{
#ifdef PLANT_TRANSPOSE
    /* wrong: dims and slots swapped inside a block */
    return ((((size_t)b * hkv + g) * bs + (size_t)(d % bs)) * dim) + (size_t)t;
#else
    return ((((size_t)b * hkv + g) * bs + t) * dim) + d;
#endif
}

/* ---------------------------------------------------------------------------
 * Slot mapping: logical position p of row r lives in slot
 * table[r][p / bs] * bs + p % bs.  Returns the number of tokens whose table
 * entry is missing or out of range (their slot is -1).
 * ------------------------------------------------------------------------- */
int32_t or_slot_mapping(const int32_t *tables, int32_t width, int32_t batch, int32_t num_blocks,
                        const int32_t *rows, const int32_t *pos, int32_t n, int32_t bs,
                        int32_t *slots)
{
    int32_t bad = 0;
    for (int32_t i = 0; i < n; ++i) {
        int32_t r = rows[i], p = pos[i];
        slots[i] = -1;
        if (r < 0 || r >= batch || p < 0 || p / bs >= width) { ++bad; continue; }
        int32_t blk = tables[(size_t)r * width + p / bs];
        if (blk < 0 || blk >= num_blocks) { ++bad; continue; }
#ifdef PLANT_SLOT
        slots[i] = blk * width + p % bs; /* wrong: table width instead of block size */
#else
        slots[i] = blk * bs + p % bs;
#endif
    }
    return bad;
}

/* ---------------------------------------------------------------------------
 * Append: copy token i's K and V rows for every kv head into its slot.
 * Storage is copied byte for byte; into an FP8 pool each bf16 element x is
 * stored as the code e4m3_encode(float32(x) / scale) (float32 division), at
 * its byte of the tile.  Returns the number of tokens skipped for a slot past
 * the pool (negative slots are skipped silently).
 * ------------------------------------------------------------------------- */
int32_t or_append(void *k_pool, void *v_pool, int32_t dtype, int32_t num_blocks, int32_t hkv,
                  int32_t bs, int32_t dim, const int32_t *slots, int32_t n, const void *k_new,
                  const void *v_new, float k_scale, float v_scale)
{
    size_t es = esize(dtype), row = (size_t)dim * es;
    int32_t bad = 0;
    if (dtype == OR_FP8 && (bs != 16 || dim % 64 != 0)) return -1;
    for (int32_t i = 0; i < n; ++i) {
        int32_t s = slots[i];
        if (s < 0) continue;
        int32_t b = s / bs, t = s % bs;
        if (b >= num_blocks) { ++bad; continue; }
        for (int32_t g = 0; g < hkv; ++g) {
#ifdef PLANT_APPEND_HEAD
            int32_t gs = (g + 1) % hkv; /* wrong: heads rotated */
#else
            int32_t gs = g;
#endif
            if (dtype == OR_FP8) {
                uint8_t *kt = (uint8_t *)k_pool + ((size_t)b * hkv + g) * (size_t)(bs * dim);
                uint8_t *vt = (uint8_t *)v_pool + ((size_t)b * hkv + g) * (size_t)(bs * dim);
                size_t src = ((size_t)i * hkv + gs) * (size_t)dim;
                for (int32_t d = 0; d < dim; ++d) {
                    float kx = (float)ld(k_new, OR_BF16, src + d);
                    float vx = (float)ld(v_new, OR_BF16, src + d);
                    kt[fp8_k_byte(t, d)] = e4m3_encode(kx / k_scale);
                    vt[fp8_v_byte(t, d)] = e4m3_encode(vx / v_scale);
                }
                continue;
            }
            size_t dst = pool_index(hkv, bs, dim, b, g, t, 0) * es;
            size_t src = ((size_t)i * hkv + gs) * row;
            memcpy((char *)k_pool + dst, (const char *)k_new + src, row);
            memcpy((char *)v_pool + dst, (const char *)v_new + src, row);
        }
    }
    return bad;
}

/* ---------------------------------------------------------------------------
 * One attention output: query vector qv (dim values at q + qoff) against the
 * keys at absolute positions lo .. hi-1 of row r, read through the row's
 * block table.  Two passes: scores and their maximum, then weights, their sum
 * and the weighted sum of values.  Returns -1 if a table entry in range is
 * missing or outside the pool (the output is then left at zero).
 * ------------------------------------------------------------------------- */
struct view {
    const void *k_pool, *v_pool;
    int32_t dtype, num_blocks, hkv, bs, dim;
    const int32_t *tables;
    int32_t width;
    double k_scale, v_scale; /* FP8 pools only */
};

/* K (is_v = 0) or V (is_v = 1) element (block b, kv head g, slot t, dim d)
 * of an FP8 pool: the code at its byte of the tile, times the pool's scale. */
static double kv_ld(const struct view *w, int is_v, int32_t b, int32_t g, int32_t t, int32_t d)
{
    const uint8_t *pool = (const uint8_t *)(is_v ? w->v_pool : w->k_pool);
    size_t tile = ((size_t)b * w->hkv + g) * (size_t)(w->bs * w->dim);
    size_t off = is_v ? fp8_v_byte(t, d) : fp8_k_byte(t, d);
    return e4m3_value(pool[tile + off]) * (is_v ? w->v_scale : w->k_scale);
}

static int attend(const struct view *w, const void *q, size_t qoff, int32_t r, int32_t g,
                  int32_t lo, int32_t hi, double scale, double *out)
{
    int32_t n = hi - lo, dim = w->dim;
    for (int32_t d = 0; d < dim; ++d) out[d] = 0.0;
    if (n <= 0) return 0;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    int32_t *blk = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    if (!s || !blk) { free(s); free(blk); return -2; }
    for (int32_t j = 0; j < n; ++j) {
        int32_t p = lo + j;
        int32_t lb = p / w->bs;
        int32_t b = (lb < w->width) ? w->tables[(size_t)r * w->width + lb] : -1;
        if (b < 0 || b >= w->num_blocks) { free(s); free(blk); return -1; }
        blk[j] = b;
    }
    double m = -INFINITY;
    for (int32_t j = 0; j < n; ++j) {
        int32_t p = lo + j;
#ifdef PLANT_OFFSET
        int32_t t = (p + 1) % w->bs; /* wrong slot inside the block */
#else
        int32_t t = p % w->bs;
#endif
        double acc = 0.0;
        if (w->dtype == OR_FP8) {
            for (int32_t d = 0; d < dim; ++d)
                acc += ld(q, OR_BF16, qoff + d) * kv_ld(w, 0, blk[j], g, t, d);
        } else {
            for (int32_t d = 0; d < dim; ++d)
                acc += ld(q, w->dtype, qoff + d) *
                       ld(w->k_pool, w->dtype, pool_index(w->hkv, w->bs, dim, blk[j], g, t, d));
        }
#ifdef PLANT_NO_SCALE
        s[j] = acc;
#else
        s[j] = scale * acc;
#endif
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int32_t j = 0; j < n; ++j) {
        double e = exp(s[j] - m);
        l += e;
        int32_t t = (lo + j) % w->bs;
#ifdef PLANT_DROP_LAST_V
        if (j == n - 1 && n > 1) continue; /* wrong: last value never accumulated */
#endif
        if (w->dtype == OR_FP8) {
            for (int32_t d = 0; d < dim; ++d) out[d] += e * kv_ld(w, 1, blk[j], g, t, d);
        } else {
            for (int32_t d = 0; d < dim; ++d)
                out[d] += e * ld(w->v_pool, w->dtype, pool_index(w->hkv, w->bs, dim, blk[j], g, t, d));
        }
    }
    for (int32_t d = 0; d < dim; ++d) out[d] /= l;
    free(s);
    free(blk);
    return 0;
}

static int32_t kv_head_of(int32_t h, int32_t hq, int32_t hkv)
{
#ifdef PLANT_GQA
    return h % hkv; /* wrong: interleaved instead of consecutive groups */
#else
    return h / (hq / hkv);
#endif
}

/* First attended position for a query at absolute position p. */
static int32_t window_lo(int32_t p, int32_t window)
{
    if (window <= 0) return 0;
#ifdef PLANT_WINDOW
    int32_t lo = p - window; /* wrong: one position too many */
#else
    int32_t lo = p - window + 1;
#endif
    return lo > 0 ? lo : 0;
}

/* ---------------------------------------------------------------------------
 * Decode: one query per row at position L-1, L = seq_lens[r].
 *   q    [batch][hq][dim]        out [batch][hq][dim] (double)
 * Returns the number of (row, head) outputs that hit a bad table entry.
 * ------------------------------------------------------------------------- */
static int decode_one(const struct view *w, const void *q, int32_t hq, const int32_t *seq_lens,
                      int32_t window, double scale, int32_t r, int32_t h, double *out)
{
    int32_t L = seq_lens[r];
    int32_t lo = L > 0 ? window_lo(L - 1, window) : 0;
    return attend(w, q, ((size_t)r * hq + h) * w->dim, r, kv_head_of(h, hq, w->hkv), lo, L,
                  scale, out);
}

int32_t or_decode(const void *q, const void *k_pool, const void *v_pool, int32_t dtype,
                  int32_t num_blocks, int32_t hq, int32_t hkv, int32_t bs, int32_t dim,
                  const int32_t *tables, int32_t width, const int32_t *seq_lens, int32_t batch,
                  int32_t window, double scale, double k_scale, double v_scale, double *out)
{
    struct view w = {k_pool, v_pool, dtype, num_blocks, hkv, bs, dim, tables, width, k_scale,
                     v_scale};
    if (dtype == OR_FP8 && (bs != 16 || dim % 64 != 0)) return -1;
    int32_t bad = 0;
    for (int32_t r = 0; r < batch; ++r)
        for (int32_t h = 0; h < hq; ++h)
            if (decode_one(&w, q, hq, seq_lens, window, scale, r, h,
                           out + ((size_t)r * hq + h) * dim))
                ++bad;
    return bad;
}

/* Decode for a list of (row, head) pairs only; out [npairs][dim]. */
int32_t or_decode_pairs(const void *q, const void *k_pool, const void *v_pool, int32_t dtype,
                        int32_t num_blocks, int32_t hq, int32_t hkv, int32_t bs, int32_t dim,
                        const int32_t *tables, int32_t width, const int32_t *seq_lens,
                        int32_t window, double scale, double k_scale, double v_scale,
                        const int32_t *rows, const int32_t *heads, int32_t npairs, double *out)
{
    struct view w = {k_pool, v_pool, dtype, num_blocks, hkv, bs, dim, tables, width, k_scale,
                     v_scale};
    if (dtype == OR_FP8 && (bs != 16 || dim % 64 != 0)) return -1;
    int32_t bad = 0;
    for (int32_t i = 0; i < npairs; ++i)
        if (decode_one(&w, q, hq, seq_lens, window, scale, rows[i], heads[i],
                       out + (size_t)i * dim))
            ++bad;
    return bad;
}

/* ---------------------------------------------------------------------------
 * Chunked prefill: row r owns queries cu[r] .. cu[r+1]-1 (C = cu[r+1]-cu[r]);
 * query i of the row sits at p_i = L - C + i and attends window_lo(p_i) .. p_i,
 * i.e. the cached prefix and the chunk's own keys up to itself.
 *   q [cu[batch]][hq][dim]       out [cu[batch]][hq][dim] (double)
 * ------------------------------------------------------------------------- */
static int prefill_one(const struct view *w, const void *q, int32_t hq, const int32_t *cu,
                       const int32_t *seq_lens, int32_t window, double scale, int32_t r,
                       int32_t i, int32_t h, double *out)
{
    int32_t c = cu[r + 1] - cu[r];
    int32_t p = seq_lens[r] - c + i;
#ifdef PLANT_CAUSAL
    int32_t hi = p + 2 <= seq_lens[r] ? p + 2 : seq_lens[r]; /* wrong: sees the next key */
#else
    int32_t hi = p + 1;
#endif
    return attend(w, q, ((size_t)(cu[r] + i) * hq + h) * w->dim, r, kv_head_of(h, hq, w->hkv),
                  window_lo(p, window), hi, scale, out);
}

int32_t or_prefill(const void *q, const int32_t *cu_q_lens, const void *k_pool,
                   const void *v_pool, int32_t dtype, int32_t num_blocks, int32_t hq, int32_t hkv,
                   int32_t bs, int32_t dim, const int32_t *tables, int32_t width,
                   const int32_t *seq_lens, int32_t batch, int32_t window, double scale,
                   double k_scale, double v_scale, double *out)
{
    struct view w = {k_pool, v_pool, dtype, num_blocks, hkv, bs, dim, tables, width, k_scale,
                     v_scale};
    if (dtype == OR_FP8 && (bs != 16 || dim % 64 != 0)) return -1;
    int32_t bad = 0;
    for (int32_t r = 0; r < batch; ++r)
        for (int32_t i = 0; i < cu_q_lens[r + 1] - cu_q_lens[r]; ++i)
            for (int32_t h = 0; h < hq; ++h)
                if (prefill_one(&w, q, hq, cu_q_lens, seq_lens, window, scale, r, i, h,
                                out + ((size_t)(cu_q_lens[r] + i) * hq + h) * dim))
                    ++bad;
    return bad;
}

/* Prefill for a list of (row, query index within the row's chunk, head). */
int32_t or_prefill_samples(const void *q, const int32_t *cu_q_lens, const void *k_pool,
                           const void *v_pool, int32_t dtype, int32_t num_blocks, int32_t hq,
                           int32_t hkv, int32_t bs, int32_t dim, const int32_t *tables,
                           int32_t width, const int32_t *seq_lens, int32_t window, double scale,
                           double k_scale, double v_scale, const int32_t *rows,
                           const int32_t *qidx, const int32_t *heads, int32_t n, double *out)
{
    struct view w = {k_pool, v_pool, dtype, num_blocks, hkv, bs, dim, tables, width, k_scale,
                     v_scale};
    if (dtype == OR_FP8 && (bs != 16 || dim % 64 != 0)) return -1;
    int32_t bad = 0;
    for (int32_t k = 0; k < n; ++k)
        if (prefill_one(&w, q, hq, cu_q_lens, seq_lens, window, scale, rows[k], qidx[k], heads[k],
                        out + (size_t)k * dim))
            ++bad;
    return bad;
}

/* ---------------------------------------------------------------------------
 * Shared-prefix groups read off the block tables ("paged-cache.md": requests
 * share refcounted blocks for a common prompt prefix; only full blocks are
 * published for reuse).  Rows whose first table entry is the same physical
 * block form a group when there are at least two of them; the group's prefix
 * is the longest run of leading entries common to all its rows, cut to the
 * blocks that are full in every row (P * bs <= L).  A group with P = 0 is
 * dropped.  Groups are numbered in the order of their lowest row.
 *   group_of_row [batch] (-1 = none), prefix_blocks [batch] (first num_groups
 *   used).  Returns num_groups.
 * ------------------------------------------------------------------------- */
int32_t or_prefix_groups(const int32_t *tables, int32_t width, const int32_t *seq_lens,
                         int32_t batch, int32_t bs, int32_t *group_of_row, int32_t *prefix_blocks)
{
    int32_t ng = 0;
    for (int32_t r = 0; r < batch; ++r) group_of_row[r] = -2; /* -2: not yet visited */
    for (int32_t r = 0; r < batch; ++r) {
        if (group_of_row[r] != -2) continue;
        int32_t first = width > 0 ? tables[(size_t)r * width] : -1;
        if (first < 0) { group_of_row[r] = -1; continue; }
        int32_t count = 0, P = width;
        for (int32_t s = r; s < batch; ++s) {
            if (group_of_row[s] != -2 || tables[(size_t)s * width] != first) continue;
            ++count;
            int32_t run = 0;
            while (run < width && tables[(size_t)s * width + run] == tables[(size_t)r * width + run])
                ++run;
#ifdef PLANT_PREFIX_CAP
            int32_t full = width;
#else
            int32_t full = seq_lens[s] / bs;
#endif
            if (run > full) run = full;
            if (run < P) P = run;
        }
        int32_t gid = (count >= 2 && P > 0) ? ng++ : -1;
        for (int32_t s = r; s < batch; ++s)
            if (group_of_row[s] == -2 && tables[(size_t)s * width] == first) group_of_row[s] = gid;
        if (gid >= 0) prefix_blocks[gid] = P;
    }
    return ng;
}
