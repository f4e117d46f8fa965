/*
 * moe_oracle.c -- plain, slow CPU oracle for the MoE decode layer with
 * host-resident cold experts.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, includes or calls
 * this file; only the tests, the smoke check and the bench's CPU-baseline leg
 * load it.  It shares no code, header, table or constant generator with the
 * CUDA path.
 *
 * Arithmetic is IEEE double throughout (inputs are bf16 activations and fp32
 * logits, both exact in double).  Every function is a direct restatement of what
 * the layer computes, step by step, with plain loops:
 *
 *   router softmax + top-k   -- "Milo and James Try Inference Engineering", the
 *                               mixture-of-experts paragraph (384 experts, a
 *                               router picks 6 per token); ties break towards the
 *                               lower expert index; weights are softmax values.
 *   bucketing                -- picks grouped by expert, stable in (token, slot).
 *   cold dedupe/remap/gather -- "DeepSeek-V4.1-Flash on One GB300 Without the
 *                               Second GPU", section 1 (The idea): one scratch slot
 *                               per cold expert, one copy of just the routed cold
 *                               experts per layer, then one call over all experts.
 *   MXFP4 decode             -- "A 475 GB Model Across Two Workstations, With the
 *                               Table on Disk", Abstract and section 1 (routed
 *                               experts ship in MXFP4); element E2M1, 32-element
 *                               blocks, E8M0 scale, per the OCP Microscaling
 *                               format the weights are named in.
 *   SwiGLU expert FFN        -- fused gate/up plane (w13) and down plane (w2),
 *                               "Milo and James Try Inference Engineering", the
 *                               offload flag table (routed_experts.w13_weight,
 *                               routed_experts.w2_weight).
 *   combine                  -- sum of router-weighted expert outputs, in pick
 *                               order ("DeepSeek-V4.1-Flash on One GB300 ...",
 *                               section 4: summation order only moves the last
 *                               decimal places).
 *   adaptive residency       -- same page, section 1 (swap often-picked cold
 *                               experts in, quiet hot ones out, between steps) and
 *                               section 3 (hysteresis threshold 3.0 as the
 *                               published default).
 *   byte audit fingerprint   -- same page, section 4 (fingerprint every expert at
 *                               boot, re-check wherever it now lives); FNV-1a 64.
 *   MXFP4 activations        -- the all-FP4 prefill mode (FP4 x FP4 tensor-core
 *                               products need both operands in MXFP4): x and h are
 *                               quantised per 32-element block by the OCP
 *                               Microscaling conversion rule and used at their
 *                               decoded values.
 *
 * Weight format (the library's documented format, restated here on its own):
 *   An expert blob is four planes, back to back:
 *     w13 nibbles [2I rows][H/2 bytes], w13 scales [2I rows][H/32 bytes],
 *     w2  nibbles [H rows][I/2 bytes],  w2  scales [H rows][I/32 bytes].
 *   Rows 0..I-1 of w13 are the gate projection, rows I..2I-1 the up projection.
 *   Scale byte (r, b) is the E8M0 exponent of block b = elements 32b..32b+31 of
 *   row r.  Inside a row, element k sits in byte k/2, in the low nibble when k is
 *   even, else the high nibble (plain K-major MXFP4 packing).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_ARG (-1)
#define OR_ERR_NONFINITE (-3)

/* ---- MXFP4 element and scale decode --------------------------------------- */

/* E2M1: sign s = bit 3, exponent field E = bits 2..1, mantissa m = bit 0.
 * E = 0 is subnormal: value m * 0.5.  Otherwise 2^(E-1) * (1 + m/2). */
double or_e2m1(unsigned code) {
    unsigned s = (code >> 3) & 1u, E = (code >> 1) & 3u, m = code & 1u;
    double mag = (E == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)E - 1);
    return s ? -mag : mag;
}

/* E8M0: 2^(e-127); e = 255 encodes NaN. */
double or_e8m0(unsigned e) {
    if (e == 255u) return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* Nibble code of element k in one row of the documented layout. */
unsigned or_nibble_at(const uint8_t* row, int k) {
    uint8_t b = row[k / 2];
    return (k % 2 == 0) ? (unsigned)(b & 0x0F) : (unsigned)(b >> 4);
}

/* Decode one row of K elements (K a multiple of 128) to doubles. */
void or_decode_row(const uint8_t* nib_row, const uint8_t* scale_row, int K, double* out) {
    for (int k = 0; k < K; ++k)
        out[k] = or_e2m1(or_nibble_at(nib_row, k)) * or_e8m0(scale_row[k / 32]);
}

/* ---- MXFP4 quantisation (all-FP4 mode) ---------------------------------------
 *
 * One block of 32 values v: with amax = max |v|, the shared exponent is
 * floor(log2(amax)) - 2 (2 = the exponent of E2M1's largest value, 6 = 1.5 * 2^2),
 * clamped to the E8M0 range [-127, 127]; the scale byte is that exponent + 127.
 * Element i is |v_i| / 2^exp rounded to the nearest E2M1 magnitude
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6}, a tie going to the even code (mantissa bit 0),
 * anything above 6 saturating to 6; the sign bit is v_i's (so -0 and negative
 * values that round to zero give code 8).  An all-zero block gets exponent -127.
 */
static const double or_e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* E2M1 code (sign bit clear) of magnitude r >= 0 by the rule above. */
static unsigned or_e2m1_round(double r) {
    if (r >= 6.0) return 7u;
    unsigned best = 0u;
    for (unsigned c = 1u; c < 8u; ++c) {
        const double dc = fabs(or_e2m1_mag[c] - r), db = fabs(or_e2m1_mag[best] - r);
        if (dc < db || (dc == db && (c & 1u) == 0u)) best = c;
    }
    return best;
}

/* Quantise K values (K a multiple of 32) into the documented row layout: K/2
 * nibble bytes (element k in byte k/2, low nibble when k is even) and K/32
 * scale bytes. */
void or_quant_mxfp4(const double* v, int K, uint8_t* nib, uint8_t* scale) {
    memset(nib, 0, (size_t)K / 2);
    for (int b = 0; b < K / 32; ++b) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs(v[32 * b + i]));
        int ex = -127;
        if (amax > 0.0) {
            int fe;
            frexp(amax, &fe); /* amax = f * 2^fe, f in [0.5, 1): floor(log2 amax) = fe - 1 */
            ex = fe - 1 - 2;
            if (ex < -127) ex = -127;
            if (ex > 127) ex = 127;
        }
        scale[b] = (uint8_t)(ex + 127);
        for (int i = 0; i < 32; ++i) {
            const int k = 32 * b + i;
            unsigned code = or_e2m1_round(ldexp(fabs(v[k]), -ex));
            if (signbit(v[k])) code |= 8u;
            nib[k / 2] |= (uint8_t)((k % 2 == 0) ? code : (code << 4));
        }
    }
}

/* v <- its MXFP4 quantisation, decoded (K a multiple of 32). */
static void or_quant_dequant(double* v, int K) {
    uint8_t* nib = (uint8_t*)malloc((size_t)K / 2);
    uint8_t* sc = (uint8_t*)malloc((size_t)K / 32);
    or_quant_mxfp4(v, K, nib, sc);
    or_decode_row(nib, sc, K, v);
    free(nib);
    free(sc);
}

/* Plane offsets of an expert blob, in bytes. */
void or_blob_offsets(int H, int I, size_t* w13n, size_t* w13s, size_t* w2n, size_t* w2s, size_t* total) {
    size_t a = (size_t)2 * I * (H / 2);
    size_t b = (size_t)2 * I * (H / 32);
    size_t c = (size_t)H * (I / 2);
    size_t d = (size_t)H * (I / 32);
    *w13n = 0;
    *w13s = a;
    *w2n = a + b;
    *w2s = a + b + c;
    *total = a + b + c + d;
}

/* bf16 bit pattern -> double (exact). */
double or_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---- router: top-k + softmax weights + bucketing --------------------------- */

/*
 * For each token t: expert e is selected iff fewer than k experts j satisfy
 * l_j > l_e, or l_j == l_e with j < e.  That count is e's rank, which is also
 * its output position (descending logit, ties to the lower index).  Weights are
 * the softmax probabilities p_e = exp(l_e - max) / sum_j exp(l_j - max) of the
 * selected experts; renorm = 1 divides them by their sum over the k picks.
 * Any non-finite logit makes the call fail with OR_ERR_NONFINITE.
 *
 * counts[e] = number of picks of e; offsets = exclusive prefix sum (E+1);
 * entries lists pick ids t*k + j grouped by expert, ascending in (t, j).
 */
int or_route(const float* logits, int T, int E, int k, int renorm,
             int32_t* ids, double* w, int32_t* counts, int32_t* offsets, int32_t* entries) {
    if (T < 0 || E <= 0 || k <= 0 || k > E) return OR_ERR_ARG;
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e)
            if (!isfinite(logits[(size_t)t * E + e])) return OR_ERR_NONFINITE;
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * E;
        for (int e = 0; e < E; ++e) {
            int rank = 0;
            for (int j = 0; j < E; ++j)
                if (l[j] > l[e] || (l[j] == l[e] && j < e)) ++rank;
            if (rank < k) ids[(size_t)t * k + rank] = e;
        }
        double mx = -INFINITY;
        for (int e = 0; e < E; ++e) mx = fmax(mx, (double)l[e]);
        double S = 0.0;
        for (int e = 0; e < E; ++e) S += exp((double)l[e] - mx);
        double sel = 0.0;
        for (int j = 0; j < k; ++j) {
            double p = exp((double)l[ids[(size_t)t * k + j]] - mx) / S;
            w[(size_t)t * k + j] = p;
            sel += p;
        }
        if (renorm)
            for (int j = 0; j < k; ++j) w[(size_t)t * k + j] /= sel;
    }
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int i = 0; i < T * k; ++i) counts[ids[i]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int pos = 0;
    for (int e = 0; e < E; ++e)
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j)
                if (ids[(size_t)t * k + j] == e) entries[pos++] = t * k + j;
    return OR_OK;
}

/* ---- placement: remap and cold gather -------------------------------------- */

/*
 * loc[e] is expert e's place: loc[e] < n_hot is an HBM slot, loc[e] = n_hot + c
 * is cold slot c (host blob c, copied into scratch slot c when routed).  The
 * physical id of a pick is loc of its expert.  cold_list gets the distinct cold
 * slots among the picks, ascending; the return value is their number.
 */
int or_remap(const int32_t* ids, int n_picks, const int32_t* loc, int n_hot, int n_cold,
             int32_t* phys, int32_t* cold_list) {
    char* seen = (char*)calloc((size_t)(n_cold > 0 ? n_cold : 1), 1);
    for (int i = 0; i < n_picks; ++i) {
        int p = loc[ids[i]];
        phys[i] = p;
        if (p >= n_hot) seen[p - n_hot] = 1;
    }
    int n = 0;
    for (int c = 0; c < n_cold; ++c)
        if (seen[c]) cold_list[n++] = c;
    free(seen);
    return n;
}

/* Byte gather with memcpy semantics: slot[c] <- host[c] for each listed c. */
void or_gather(uint8_t* const* slots, const uint8_t* const* host, const int32_t* cold_list, int n,
               size_t blob_bytes) {
    for (int i = 0; i < n; ++i) memcpy(slots[cold_list[i]], host[cold_list[i]], blob_bytes);
}

/* ---- expert FFN ------------------------------------------------------------- */

/*
 * One expert on n_tok tokens.  x: [n_tok][H] doubles; y: [n_tok][H] doubles.
 *   g = W_gate x, u = W_up x       (w13 rows 0..I-1 and I..2I-1)
 *   h = SiLU(g) * u, SiLU(g) = g / (1 + exp(-g))
 *   y = W2 h                       (w2 is [H rows][I columns])
 * Dot products run in index order.
 */
/* act4 = 1: the all-FP4 mode -- each token's x row is quantised to MXFP4 (blocks
 * along H) and each token's h row (blocks along I) before it meets W2. */
static void or_expert_ffn_mode(const uint8_t* blob, int H, int I, const double* x_in, int n_tok, double* y,
                               int act4) {
    size_t o13n, o13s, o2n, o2s, tot;
    or_blob_offsets(H, I, &o13n, &o13s, &o2n, &o2s, &tot);
    double* row = (double*)malloc(sizeof(double) * (size_t)(H > I ? H : I));
    double* row2 = (double*)malloc(sizeof(double) * (size_t)H);
    double* h = (double*)malloc(sizeof(double) * (size_t)n_tok * I);
    double* xq = (double*)malloc(sizeof(double) * (size_t)n_tok * H);
    memcpy(xq, x_in, sizeof(double) * (size_t)n_tok * H);
    if (act4)
        for (int t = 0; t < n_tok; ++t) or_quant_dequant(xq + (size_t)t * H, H);
    const double* x = xq;
    for (int r = 0; r < I; ++r) {
        or_decode_row(blob + o13n + (size_t)r * (H / 2), blob + o13s + (size_t)r * (H / 32), H, row);
        or_decode_row(blob + o13n + (size_t)(I + r) * (H / 2), blob + o13s + (size_t)(I + r) * (H / 32), H, row2);
        for (int t = 0; t < n_tok; ++t) {
            double g = 0.0, u = 0.0;
            for (int c = 0; c < H; ++c) {
                g += row[c] * x[(size_t)t * H + c];
                u += row2[c] * x[(size_t)t * H + c];
            }
            h[(size_t)t * I + r] = g / (1.0 + exp(-g)) * u;
        }
    }
    if (act4)
        for (int t = 0; t < n_tok; ++t) or_quant_dequant(h + (size_t)t * I, I);
    for (int r = 0; r < H; ++r) {
        or_decode_row(blob + o2n + (size_t)r * (I / 2), blob + o2s + (size_t)r * (I / 32), I, row);
        for (int t = 0; t < n_tok; ++t) {
            double acc = 0.0;
            for (int c = 0; c < I; ++c) acc += row[c] * h[(size_t)t * I + c];
            y[(size_t)t * H + r] = acc;
        }
    }
    free(row);
    free(row2);
    free(h);
    free(xq);
}

void or_expert_ffn(const uint8_t* blob, int H, int I, const double* x, int n_tok, double* y) {
    or_expert_ffn_mode(blob, H, I, x, n_tok, y, 0);
}

void or_expert_ffn_act4(const uint8_t* blob, int H, int I, const double* x, int n_tok, double* y) {
    or_expert_ffn_mode(blob, H, I, x, n_tok, y, 1);
}

/* out[t][c] = sum over j = 0..k-1 (in order) of w[t][j] * y[t*k + j][c]. */
void or_combine(const double* y, const double* w, int T, int k, int H, double* out) {
    for (int t = 0; t < T; ++t)
        for (int c = 0; c < H; ++c) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) acc += w[(size_t)t * k + j] * y[((size_t)t * k + j) * H + c];
            out[(size_t)t * H + c] = acc;
        }
}

/*
 * Whole layer for T tokens: route, then every pick's expert FFN on its token
 * (blobs[e] points at expert e's bytes, wherever they live), then combine.
 * x_bf16: [T][H] bf16 bits.  Outputs ids/w/out; y is scratch [T*k][H].
 */
static int or_layer_mode(const float* logits, const uint16_t* x_bf16, int T, int E, int k, int renorm, int H, int I,
                         const uint8_t* const* blobs, int32_t* ids, double* w, double* out, int act4) {
    int32_t* counts = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    int32_t* entries = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T * k > 0 ? T * k : 1));
    int rc = or_route(logits, T, E, k, renorm, ids, w, counts, offsets, entries);
    if (rc != OR_OK) {
        free(counts); free(offsets); free(entries);
        return rc;
    }
    double* x = (double*)malloc(sizeof(double) * (size_t)H);
    double* y = (double*)malloc(sizeof(double) * (size_t)(T * k > 0 ? T * k : 1) * H);
    for (int t = 0; t < T; ++t) {
        for (int c = 0; c < H; ++c) x[c] = or_bf16(x_bf16[(size_t)t * H + c]);
        for (int j = 0; j < k; ++j)
            or_expert_ffn_mode(blobs[ids[(size_t)t * k + j]], H, I, x, 1, y + ((size_t)t * k + j) * H, act4);
    }
    or_combine(y, w, T, k, H, out);
    free(x); free(y); free(counts); free(offsets); free(entries);
    return OR_OK;
}

int or_layer(const float* logits, const uint16_t* x_bf16, int T, int E, int k, int renorm, int H, int I,
             const uint8_t* const* blobs, int32_t* ids, double* w, double* out) {
    return or_layer_mode(logits, x_bf16, T, E, k, renorm, H, I, blobs, ids, w, out, 0);
}

/* The whole layer in the all-FP4 mode (or_expert_ffn_act4 for every pick). */
int or_layer_act4(const float* logits, const uint16_t* x_bf16, int T, int E, int k, int renorm, int H, int I,
                  const uint8_t* const* blobs, int32_t* ids, double* w, double* out) {
    return or_layer_mode(logits, x_bf16, T, E, k, renorm, H, I, blobs, ids, w, out, 1);
}

/* ---- adaptive residency ------------------------------------------------------ */

static const int32_t* g_cnt; /* qsort context */

static int cmp_cold(const void* a, const void* b) { /* count desc, id asc */
    int x = *(const int*)a, y = *(const int*)b;
    if (g_cnt[x] != g_cnt[y]) return g_cnt[x] > g_cnt[y] ? -1 : 1;
    return x < y ? -1 : (x > y);
}

static int cmp_hot(const void* a, const void* b) { /* count asc, id asc */
    int x = *(const int*)a, y = *(const int*)b;
    if (g_cnt[x] != g_cnt[y]) return g_cnt[x] < g_cnt[y] ? -1 : 1;
    return x < y ? -1 : (x > y);
}

/*
 * One residency update from the pick counts of the window just ended.
 * Candidates: cold experts picked at least once (count desc, id asc) and hot
 * experts (count asc, id asc).  Pair them in order; pair i swaps when
 * count(cold_i) > hysteresis * count(hot_i), and the first pair that fails
 * ends the update; at most max_swaps pairs.  A swap exchanges the two experts'
 * places: the promoted one takes the demoted one's HBM slot, the demoted one
 * takes the promoted one's cold slot.  loc is updated in place; promoted[i] and
 * demoted[i] list the swapped experts in order; the return value is the count.
 */
int or_residency(const int32_t* counts, int32_t* loc, int E, int n_hot, int max_swaps, double hysteresis,
                 int32_t* promoted, int32_t* demoted) {
    int* cold = (int*)malloc(sizeof(int) * (size_t)E);
    int* hot = (int*)malloc(sizeof(int) * (size_t)E);
    int nc = 0, nh = 0;
    for (int e = 0; e < E; ++e) {
        if (loc[e] >= n_hot) {
            if (counts[e] >= 1) cold[nc++] = e;
        } else {
            hot[nh++] = e;
        }
    }
    g_cnt = counts;
    qsort(cold, (size_t)nc, sizeof(int), cmp_cold);
    qsort(hot, (size_t)nh, sizeof(int), cmp_hot);
    int lim = max_swaps;
    if (nc < lim) lim = nc;
    if (nh < lim) lim = nh;
    int n = 0;
    for (int i = 0; i < lim; ++i) {
        int a = cold[i], b = hot[i];
        if (!((double)counts[a] > hysteresis * (double)counts[b])) break;
        int tmp = loc[a];
        loc[a] = loc[b];
        loc[b] = tmp;
        promoted[n] = a;
        demoted[n] = b;
        ++n;
    }
    free(cold);
    free(hot);
    return n;
}

/* ---- byte audit --------------------------------------------------------------- */

uint64_t or_fnv1a64(const uint8_t* p, size_t n) {
    uint64_t h = 0xcbf29ce484222325ull;
    for (size_t i = 0; i < n; ++i) {
        h ^= (uint64_t)p[i];
        h *= 0x100000001b3ull;
    }
    return h;
}
