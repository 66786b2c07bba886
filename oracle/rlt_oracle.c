/*
 * CPU oracle for the paged decode path of looped transformers.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline of the benchmark may load this file's library.  It shares no code,
 * header, table or constant generator with the CUDA library: it is a plain,
 * slow, single-threaded restatement of what the path computes, in fp64 for
 * all floating point.
 *
 * Sources (page title, section):
 *   [FFM]   "Faster fuzzy minds" (dibbla.space), sections "When scheduler does
 *           the work" (paged KV cache: flat pool of slots addressed through
 *           page_table[request, position]), "LOTUS - the one place I opened the
 *           scheduler" (store_kv scatters each token's K/V to the slots it is
 *           handed), "Recurrent depth - a deep model in a trench coat"
 *           (iteration t, layer l writes KV bank t*L + l).
 *   [PR152] vllm-rlt PR #152 "[Huginn] Opt-in prefix caching with
 *           position-keyed recurrent-state noise", section Summary, paragraphs
 *           1 and 2 (per-plane layer map of #147; noise as a function of
 *           (request seed, position, channel) through a stage-wise
 *           SplitMix64-style hash, a 24-bit uniform and an inverse normal CDF
 *           onto a normal truncated at +-3 sigma with std = initializer_range).
 *
 * Pool layout (the library's documented layout, an input convention, not an
 * algorithm): K and V are separate arrays of bf16 bit patterns laid out
 * [bank][page][kv_head][offset in page][head_dim].  A token at logical
 * position p of request b lives at page page_table[b][p / page_size], offset
 * p % page_size.
 *
 * Parity pins for every function here live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---------------------------------------------------------------- helpers */

static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;     /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int64_t pool_row(int64_t bank, int64_t page, int64_t head, int64_t offset,
                        int64_t num_pages, int64_t num_kv_heads, int64_t page_size,
                        int64_t head_dim)
{
    return (((bank * num_pages + page) * num_kv_heads + head) * page_size + offset) * head_dim;
}

/* ------------------------------------------------------ bank map [PR152] */

/*
 * Bank of every (layer, plane): map[layer * num_planes + plane], -1 where the
 * plane does not hold the layer.  Plane 0 holds every layer; deeper planes
 * hold only the looped (recurrent) layers ("all layers at depth 0, the
 * recurrent layers deeper", [PR152] Summary para 1).  Banks are numbered plane
 * by plane, layers in order inside a plane, so a fully looped stack gets bank
 * t*L + l exactly as in [FFM] "Recurrent depth".  Returns the bank count.
 */
int32_t oracle_bank_map(const uint8_t *recurrent, int32_t num_layers, int32_t num_planes,
                        int32_t *map)
{
    int32_t next = 0;
    for (int32_t plane = 0; plane < num_planes; ++plane)
        for (int32_t layer = 0; layer < num_layers; ++layer) {
            int held = (plane == 0) || recurrent[layer];
            map[layer * num_planes + plane] = held ? next++ : -1;
        }
    return next;
}

/* ---------------------------------------------- slot of a token [FFM] */

/* Physical slot of logical position pos of request b: page * page_size + offset. */
int64_t oracle_slot(const int32_t *page_table, int32_t max_pages, int32_t b, int64_t pos,
                    int32_t page_size)
{
    int64_t page = page_table[(int64_t)b * max_pages + pos / page_size];
    return page * page_size + pos % page_size;
}

/*
 * Gather every request's cached K and V rows, in logical order, into dense
 * [B][max_len][Hkv][D] arrays (bf16 bits, copied unchanged).  Rows at or past
 * a request's length are left as they are.
 */
void oracle_paged_gather(const uint16_t *k_pool, const uint16_t *v_pool, int64_t num_pages,
                         int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                         int32_t bank, const int32_t *page_table, int32_t max_pages,
                         const int32_t *seq_lens, int32_t batch, int32_t max_len,
                         uint16_t *k_out, uint16_t *v_out)
{
    for (int32_t b = 0; b < batch; ++b)
        for (int64_t pos = 0; pos < seq_lens[b]; ++pos) {
            int64_t slot = oracle_slot(page_table, max_pages, b, pos, page_size);
            int64_t page = slot / page_size, offset = slot % page_size;
            for (int32_t g = 0; g < num_kv_heads; ++g) {
                int64_t src = pool_row(bank, page, g, offset, num_pages, num_kv_heads,
                                       page_size, head_dim);
                int64_t dst = (((int64_t)b * max_len + pos) * num_kv_heads + g) * head_dim;
                for (int32_t d = 0; d < head_dim; ++d) {
                    k_out[dst + d] = k_pool[src + d];
                    v_out[dst + d] = v_pool[src + d];
                }
            }
        }
}

/* -------------------------------------------------- KV append [FFM] LOTUS */

/*
 * store_kv: write token i's K and V rows ([Hkv][D] each) to slot out_loc[i]
 * of the given bank, in place.  Slots below zero are skipped (no token).
 * Writing the same slots again overwrites them (LOTUS in-place re-forward).
 */
void oracle_kv_append(uint16_t *k_pool, uint16_t *v_pool, int64_t num_pages,
                      int32_t num_kv_heads, int32_t page_size, int32_t head_dim, int32_t bank,
                      const uint16_t *k_new, const uint16_t *v_new, const int64_t *out_loc,
                      int32_t n_tokens)
{
    for (int32_t i = 0; i < n_tokens; ++i) {
        int64_t slot = out_loc[i];
        if (slot < 0)
            continue;
        int64_t page = slot / page_size, offset = slot % page_size;
        for (int32_t g = 0; g < num_kv_heads; ++g) {
            int64_t dst = pool_row(bank, page, g, offset, num_pages, num_kv_heads, page_size,
                                   head_dim);
            int64_t src = ((int64_t)i * num_kv_heads + g) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) {
                k_pool[dst + d] = k_new[src + d];
                v_pool[dst + d] = v_new[src + d];
            }
        }
    }
}

/* ------------------------------------------ paged decode attention [FFM] */

/*
 * One query token per request attends over all seq_lens[b] cached tokens of
 * its request, gathered through the page table:
 *     s_j = scale * <q_h, k_j>,   o_h = sum_j softmax(s)_j v_j,
 * query head h reading kv head h / (Hq / Hkv) (consecutive GQA groups).
 * lse[b][h] = log sum_j exp(s_j) (natural log).  A request with no cached
 * token gets o = 0 and lse = -inf.  scale <= 0 means 1 / sqrt(head_dim).
 * All arithmetic in fp64 on the exact bf16 input values.
 */
void oracle_decode_attn(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                        int64_t num_pages, int32_t num_kv_heads, int32_t page_size,
                        int32_t head_dim, int32_t bank, const int32_t *page_table,
                        int32_t max_pages, const int32_t *seq_lens, int32_t batch,
                        int32_t num_q_heads, double scale, double *out, double *lse,
                        double *scores /* workspace, >= max seq_len doubles */)
{
    if (scale <= 0)
        scale = 1.0 / sqrt((double)head_dim);
    int32_t group = num_q_heads / num_kv_heads;
    for (int32_t b = 0; b < batch; ++b) {
        int64_t L = seq_lens[b];
        for (int32_t h = 0; h < num_q_heads; ++h) {
            int32_t g = h / group;
            const uint16_t *qh = q + ((int64_t)b * num_q_heads + h) * head_dim;
            double *oh = out + ((int64_t)b * num_q_heads + h) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d)
                oh[d] = 0.0;
            if (L == 0) {
                lse[(int64_t)b * num_q_heads + h] = -INFINITY;
                continue;
            }
            double m = -INFINITY;
            for (int64_t j = 0; j < L; ++j) {
                int64_t slot = oracle_slot(page_table, max_pages, b, j, page_size);
                int64_t row = pool_row(bank, slot / page_size, g, slot % page_size, num_pages,
                                       num_kv_heads, page_size, head_dim);
                double dot = 0.0;
                for (int32_t d = 0; d < head_dim; ++d)
                    dot += bf16_value(qh[d]) * bf16_value(k_pool[row + d]);
                scores[j] = scale * dot;
                if (scores[j] > m)
                    m = scores[j];
            }
            double denom = 0.0;
            for (int64_t j = 0; j < L; ++j) {
                int64_t slot = oracle_slot(page_table, max_pages, b, j, page_size);
                int64_t row = pool_row(bank, slot / page_size, g, slot % page_size, num_pages,
                                       num_kv_heads, page_size, head_dim);
                double w = exp(scores[j] - m);
                denom += w;
                for (int32_t d = 0; d < head_dim; ++d)
                    oh[d] += w * bf16_value(v_pool[row + d]);
            }
            for (int32_t d = 0; d < head_dim; ++d)
                oh[d] /= denom;
            lse[(int64_t)b * num_q_heads + h] = m + log(denom);
        }
    }
}

/* --------------------------------------- position-keyed noise [PR152] */

/* SplitMix64 output function (Steele, Lea & Flood, OOPSLA 2014), mod 2^64. */
uint64_t oracle_mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * UINT64_C(0xBF58476D1CE4E5B9);
    z = (z ^ (z >> 27)) * UINT64_C(0x94D049BB133111EB);
    return z ^ (z >> 31);
}

/* One stage: fold key x into state h, advance by the golden-ratio increment, mix. */
uint64_t oracle_stage(uint64_t h, uint64_t x)
{
    return oracle_mix64((h ^ x) + UINT64_C(0x9E3779B97F4A7C15));
}

/* Stage-wise key: request seed, then absolute position, then channel. */
uint64_t oracle_noise_key(uint64_t seed, int64_t position, int32_t channel)
{
    uint64_t h = oracle_stage(0, seed);
    h = oracle_stage(h, (uint64_t)position);
    return oracle_stage(h, (uint64_t)(int64_t)channel);
}

/* The 24-bit uniform: the top 24 bits of the key. */
void oracle_noise_hash24(const uint64_t *seeds, const int64_t *positions, int64_t n_rows,
                         int32_t channels, uint32_t *out)
{
    for (int64_t r = 0; r < n_rows; ++r)
        for (int32_t c = 0; c < channels; ++c)
            out[r * channels + c] = (uint32_t)(oracle_noise_key(seeds[r], positions[r], c) >> 40);
}

/* Standard normal CDF from the C library's complementary error function. */
static double normal_cdf(double x)
{
    return 0.5 * erfc(-x / sqrt(2.0));
}

/* Inverse standard normal CDF on (Phi(-3), Phi(3)) by bisection on [-3, 3]. */
static double normal_cdf_inverse(double p)
{
    double lo = -3.0, hi = 3.0;
    for (int it = 0; it < 200; ++it) {
        double mid = 0.5 * (lo + hi);
        if (mid <= lo || mid >= hi)
            break;                          /* interval is one ulp wide */
        if (normal_cdf(mid) < p)
            lo = mid;
        else
            hi = mid;
    }
    return 0.5 * (lo + hi);
}

/*
 * Truncated-normal value of one 24-bit uniform: u = (h24 + 1/2) / 2^24 is the
 * midpoint of the h24-th of 2^24 equal cells of (0, 1); the inverse CDF of
 * N(0, 1) truncated to [-3, 3] is Phi^-1(Phi(-3) + u (Phi(3) - Phi(-3))); the
 * value is that times sigma = initializer_range.
 */
double oracle_noise_value(uint32_t h24, double initializer_range)
{
    double u = ((double)h24 + 0.5) / 16777216.0;
    double lo = normal_cdf(-3.0), hi = normal_cdf(3.0);
    return initializer_range * normal_cdf_inverse(lo + u * (hi - lo));
}

/* Initial latent state x[r][c] of every row (token) and channel, in fp64. */
void oracle_latent_noise_init(const uint64_t *seeds, const int64_t *positions, int64_t n_rows,
                              int32_t channels, double initializer_range, double *out)
{
    for (int64_t r = 0; r < n_rows; ++r)
        for (int32_t c = 0; c < channels; ++c) {
            uint32_t h24 = (uint32_t)(oracle_noise_key(seeds[r], positions[r], c) >> 40);
            out[r * channels + c] = oracle_noise_value(h24, initializer_range);
        }
}

/* ------------------------------------------- RoPE at the token's position */

/*
 * Correctly rounded (nearest, ties to even) bf16 bit pattern of a double: the
 * value is scaled by the bf16 quantum of its binade (a power of two, so the
 * scaling is exact), rounded to an integer, and scaled back.
 */
static uint16_t bf16_round(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (ax == 0.0)
        return sign;
    int e;
    frexp(ax, &e);                        /* ax = m * 2^e, m in [1/2, 1) */
    int qe = e - 8;                       /* 8 significant bits */
    if (qe < -133)
        qe = -133;                        /* subnormal quantum 2^-133 */
    double r = rint(ldexp(ax, -qe));      /* default rounding: nearest, ties to even */
    double v = ldexp(r, qe);
    if (v >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80); /* overflow: infinity */
    float f = (float)v;                   /* exact: v has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

uint16_t oracle_bf16_round(double x) { return bf16_round(x); }

/*
 * Rotary position embedding of one head row x[head_dim] at sequence position
 * pos, as the fused append applies it to keys.  [FFM] "Recurrent depth": a
 * token keeps one RoPE position across all T of its banks, so pos is the
 * token's index in its sequence, never its loop depth.  Rotate-half pairing:
 * for i < rot_dim / 2 the pair (x[i], x[i + rot_dim/2]) turns by the angle
 * pos * base^(-2i / rot_dim); dims rot_dim .. head_dim-1 are copied.  fp64.
 */
void oracle_rope(const double *x, int32_t head_dim, int32_t rot_dim, double base, int64_t pos,
                 double *out)
{
    int32_t half = rot_dim / 2;
    for (int32_t d = 0; d < head_dim; ++d)
        out[d] = x[d];
    for (int32_t i = 0; i < half; ++i) {
        double angle = (double)pos * pow(base, -2.0 * i / rot_dim);
        double c = cos(angle), s = sin(angle);
        out[i] = x[i] * c - x[i + half] * s;
        out[i + half] = x[i] * s + x[i + half] * c;
    }
}

/*
 * store_kv with the keys rotated first: token i's K rows (bf16 [Hkv][D]) turn
 * by RoPE at positions[i] and are rounded to bf16 (nearest even); its V rows
 * are copied.  Written to slot out_loc[i] of the bank; slots below zero are
 * skipped.
 */
void oracle_kv_append_rope(uint16_t *k_pool, uint16_t *v_pool, int64_t num_pages,
                           int32_t num_kv_heads, int32_t page_size, int32_t head_dim, int32_t bank,
                           const uint16_t *k_new, const uint16_t *v_new, const int64_t *positions,
                           const int64_t *out_loc, int32_t n_tokens, int32_t rot_dim, double base)
{
    double x[1024], y[1024];
    if (head_dim > 1024)
        return;
    for (int32_t i = 0; i < n_tokens; ++i) {
        int64_t slot = out_loc[i];
        if (slot < 0)
            continue;
        int64_t page = slot / page_size, offset = slot % page_size;
        for (int32_t g = 0; g < num_kv_heads; ++g) {
            int64_t dst = pool_row(bank, page, g, offset, num_pages, num_kv_heads, page_size,
                                   head_dim);
            int64_t src = ((int64_t)i * num_kv_heads + g) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d)
                x[d] = bf16_value(k_new[src + d]);
            oracle_rope(x, head_dim, rot_dim, base, positions[i], y);
            for (int32_t d = 0; d < head_dim; ++d) {
                k_pool[dst + d] = bf16_round(y[d]);
                v_pool[dst + d] = v_new[src + d];
            }
        }
    }
}

/* --------------------------------------- prefix publication [PR152] */

/*
 * Written-prefix counters: written[bank * batch + r] is the length of the
 * prefix of request r that the bank holds.  Appends come in sequence order
 * (a decode token, or a prefill chunk), so each appended token at position p
 * extends the counter to at least p + 1.  Tokens with out_loc < 0 are skipped.
 */
void oracle_mark_written(int32_t *written, int32_t batch, int32_t bank, const int32_t *request,
                         const int64_t *positions, const int64_t *out_loc, int32_t n_tokens)
{
    for (int32_t i = 0; i < n_tokens; ++i) {
        if (out_loc[i] < 0)
            continue;
        int32_t *w = &written[(int64_t)bank * batch + request[i]];
        if (*w < positions[i] + 1)
            *w = (int32_t)(positions[i] + 1);
    }
}

/*
 * Tokens of each request that may be published to the prefix cache: the
 * prefix written in every (layer, plane) bank the model holds, in whole pages.
 * [PR152] Summary (per-plane coverage, "all layers at depth 0, the recurrent
 * layers deeper"): planes that do not hold a layer (map -1) are not asked for
 * it.  A model holding no bank publishes nothing.
 */
void oracle_publishable_prefix(const int32_t *map, int32_t num_layers, int32_t num_planes,
                               const int32_t *written, int32_t batch, int32_t page_size,
                               int32_t *out)
{
    for (int32_t b = 0; b < batch; ++b) {
        int64_t m = -1;
        for (int32_t l = 0; l < num_layers; ++l)
            for (int32_t t = 0; t < num_planes; ++t) {
                int32_t bank = map[l * num_planes + t];
                if (bank < 0)
                    continue;
                int64_t w = written[(int64_t)bank * batch + b];
                if (m < 0 || w < m)
                    m = w;
            }
        out[b] = m < 0 ? 0 : (int32_t)(m / page_size * page_size);
    }
}
