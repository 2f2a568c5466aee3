/*
 * CPU oracle for the submanifold sparse 3-D convolution.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * What it computes, and where that is defined (page: "sparse_conv_metal.py",
 * trellis-2-mrp-mlx, mlx_backend):
 *
 *   oracle_build_nmap  the neighbour map the page's kernel consumes: a (K, N)
 *                      int32 array, entry [k, n] = index of the active voxel
 *                      at coords[n] + offsets[k], or N when there is none
 *                      (the wrapper docstring fixes the shape, the int32 type
 *                      and N as the marker of a missing neighbour; the page
 *                      does not show how the map is built, so this is the
 *                      plain definition: sort the packed coordinates and
 *                      binary-search every neighbour).
 *
 *   oracle_conv        out[n, co] = bias[co] + sum_k sum_ci
 *                          feats[nmap[k, n], ci] * w[k, ci, co]
 *                      (module docstring formula; kernel body: skip an entry
 *                      that is not a valid row, accumulate over k then ci;
 *                      wrapper: bias added to the result).  Accumulation is
 *                      in double precision over the stored values widened
 *                      exactly, so the result is the exact sum up to fp64
 *                      rounding.  It also returns sabs[n, co] = |bias[co]| +
 *                      sum |term|, the scale the acceptance tolerance is
 *                      measured against.
 *
 *   oracle_dgrad       d out / d feats, the adjoint of the formula above:
 *                      dfeats[m, ci] = sum over valid entries m = nmap[k, n]
 *                      of sum_co dout[n, co] * w[k, ci, co].
 *   oracle_wgrad       d out / d w: dw[k, ci, co] = sum over valid entries
 *                      of feats[nmap[k, n], ci] * dout[n, co].
 *                      The page computes the forward pass only; these two
 *                      are the chain rule applied to its formula, written
 *                      out as plain sums in fp64 (with sum |term| scales).
 *
 * Readings where the page is silent: a neighbour lies at coords[n] +
 * offsets[k] (cross-correlation); an entry is valid iff 0 <= v < N (the page
 * skips v >= N; negative values are treated the same way instead of being
 * read); coordinates are unique and each component lies in [0, 2^20).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_INVALID_ARG (-1)
#define ORACLE_ERR_DUPLICATE_COORD (-4)
#define ORACLE_ERR_NOMEM (-6)

#define ORACLE_DTYPE_F32 0  /* fp32 storage */
#define ORACLE_DTYPE_BF16 1 /* bfloat16 storage (uint16 bit patterns) */

#define COORD_LIMIT (1 << 20)

typedef struct {
    uint64_t key;
    int64_t index;
} oracle_entry;

static int oracle_in_range(int64_t v) { return v >= 0 && v < COORD_LIMIT; }

static uint64_t oracle_pack(int64_t z, int64_t y, int64_t x)
{
    return ((uint64_t)z << 40) | ((uint64_t)y << 20) | (uint64_t)x;
}

static int oracle_cmp_entry(const void* a, const void* b)
{
    uint64_t ka = ((const oracle_entry*)a)->key;
    uint64_t kb = ((const oracle_entry*)b)->key;
    return (ka > kb) - (ka < kb);
}

/* Sorted (key, index) table of all voxels; NULL on allocation failure.
 * *status is set to ORACLE_ERR_DUPLICATE_COORD when two voxels share a key. */
static oracle_entry* oracle_sorted_table(const int32_t* coords, int64_t N, int* status)
{
    oracle_entry* table = (oracle_entry*)malloc((size_t)N * sizeof(oracle_entry));
    *status = ORACLE_OK;
    if (table == NULL) {
        *status = ORACLE_ERR_NOMEM;
        return NULL;
    }
    for (int64_t n = 0; n < N; ++n) {
        table[n].key = oracle_pack(coords[3 * n], coords[3 * n + 1], coords[3 * n + 2]);
        table[n].index = n;
    }
    qsort(table, (size_t)N, sizeof(oracle_entry), oracle_cmp_entry);
    for (int64_t i = 1; i < N; ++i) {
        if (table[i].key == table[i - 1].key) {
            free(table);
            *status = ORACLE_ERR_DUPLICATE_COORD;
            return NULL;
        }
    }
    return table;
}

/* Index of the voxel at coords[n] + offsets[k], or N. */
static int32_t oracle_neighbour(const oracle_entry* table, const int32_t* coords, int64_t N,
                                const int32_t* offsets, int64_t n, int32_t k)
{
    int64_t z = (int64_t)coords[3 * n] + offsets[3 * k];
    int64_t y = (int64_t)coords[3 * n + 1] + offsets[3 * k + 1];
    int64_t x = (int64_t)coords[3 * n + 2] + offsets[3 * k + 2];
    if (!(oracle_in_range(z) && oracle_in_range(y) && oracle_in_range(x))) return (int32_t)N;
    oracle_entry probe;
    probe.key = oracle_pack(z, y, x);
    probe.index = 0;
    const oracle_entry* hit = (const oracle_entry*)bsearch(&probe, table, (size_t)N,
                                                           sizeof(oracle_entry), oracle_cmp_entry);
    return hit != NULL ? (int32_t)hit->index : (int32_t)N;
}

static int oracle_check_coords(const int32_t* coords, int64_t N)
{
    for (int64_t n = 0; n < N; ++n)
        for (int c = 0; c < 3; ++c)
            if (!oracle_in_range(coords[3 * n + c])) return ORACLE_ERR_INVALID_ARG;
    return ORACLE_OK;
}

/* Neighbour map by sort + binary search: nmap is (K, N).  Returns ORACLE_OK
 * or an error. */
int oracle_build_nmap(const int32_t* coords, int64_t N, const int32_t* offsets, int32_t K,
                      int32_t* nmap)
{
    if (N < 0 || K < 1 || (N > 0 && (coords == NULL || nmap == NULL)) || offsets == NULL)
        return ORACLE_ERR_INVALID_ARG;
    if (N >= INT32_MAX) return ORACLE_ERR_INVALID_ARG;
    if (N == 0) return ORACLE_OK;
    int status = oracle_check_coords(coords, N);
    if (status != ORACLE_OK) return status;
    oracle_entry* table = oracle_sorted_table(coords, N, &status);
    if (table == NULL) return status;
    for (int64_t n = 0; n < N; ++n)
        for (int32_t k = 0; k < K; ++k)
            nmap[(size_t)k * (size_t)N + (size_t)n] = oracle_neighbour(table, coords, N, offsets, n, k);
    free(table);
    return ORACLE_OK;
}

/* The same map restricted to the voxels rows[0 .. n_rows): out is (K, n_rows),
 * out[k, r] = nmap[k, rows[r]]. */
int oracle_nmap_rows(const int32_t* coords, int64_t N, const int32_t* offsets, int32_t K,
                     const int64_t* rows, int64_t n_rows, int32_t* out)
{
    if (N < 1 || K < 1 || coords == NULL || offsets == NULL || rows == NULL || out == NULL ||
        n_rows < 0 || N >= INT32_MAX)
        return ORACLE_ERR_INVALID_ARG;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return ORACLE_ERR_INVALID_ARG;
    int status = oracle_check_coords(coords, N);
    if (status != ORACLE_OK) return status;
    oracle_entry* table = oracle_sorted_table(coords, N, &status);
    if (table == NULL) return status;
    for (int64_t r = 0; r < n_rows; ++r)
        for (int32_t k = 0; k < K; ++k)
            out[(size_t)k * (size_t)n_rows + (size_t)r] =
                oracle_neighbour(table, coords, N, offsets, rows[r], k);
    free(table);
    return ORACLE_OK;
}

/*
 * The same map in pieces, for large inputs split over host threads: the
 * sorted table is built once (oracle_table_new) and each caller fills the
 * columns n0 <= n < n1 of the full (K, N) map with the same binary search
 * (oracle_table_query); oracle_table_free releases the table.
 */
void* oracle_table_new(const int32_t* coords, int64_t N, int* status)
{
    if (status == NULL) return NULL;
    if (N < 1 || coords == NULL || N >= INT32_MAX) {
        *status = ORACLE_ERR_INVALID_ARG;
        return NULL;
    }
    *status = oracle_check_coords(coords, N);
    if (*status != ORACLE_OK) return NULL;
    return oracle_sorted_table(coords, N, status);
}

int oracle_table_query(const void* table, const int32_t* coords, int64_t N, const int32_t* offsets,
                       int32_t K, int64_t n0, int64_t n1, int32_t* nmap)
{
    if (table == NULL || coords == NULL || offsets == NULL || nmap == NULL || K < 1 || n0 < 0 ||
        n1 > N || n0 > n1)
        return ORACLE_ERR_INVALID_ARG;
    for (int64_t n = n0; n < n1; ++n)
        for (int32_t k = 0; k < K; ++k)
            nmap[(size_t)k * (size_t)N + (size_t)n] =
                oracle_neighbour((const oracle_entry*)table, coords, N, offsets, n, k);
    return ORACLE_OK;
}

void oracle_table_free(void* table) { free(table); }

/* Exact widening of one stored value to double. */
static double oracle_widen(const void* base, int32_t dtype, size_t i)
{
    if (dtype == ORACLE_DTYPE_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[i];
}

/*
 * The convolution, plain loop nest in fp64.  Computes the output rows listed
 * in rows[0 .. n_rows) (all N rows in order when rows == NULL), writing
 * out[r * Co + co] and sabs[r * Co + co] for the r-th listed row.
 * bias may be NULL (treated as zero).
 */
int oracle_conv(const void* feats, int32_t dtype, const int32_t* nmap, const void* w,
                const void* bias, int64_t N, int32_t K, int32_t Ci, int32_t Co,
                const int64_t* rows, int64_t n_rows, double* out, double* sabs)
{
    if (N < 1 || K < 1 || Ci < 1 || Co < 1 || feats == NULL || nmap == NULL || w == NULL ||
        out == NULL || sabs == NULL)
        return ORACLE_ERR_INVALID_ARG;
    if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return ORACLE_ERR_INVALID_ARG;
    int64_t count = rows != NULL ? n_rows : N;

    for (int64_t r = 0; r < count; ++r) {
        int64_t n = rows != NULL ? rows[r] : r;
        if (n < 0 || n >= N) return ORACLE_ERR_INVALID_ARG;
        for (int32_t co = 0; co < Co; ++co) {
            double acc = bias != NULL ? oracle_widen(bias, dtype, (size_t)co) : 0.0;
            double mag = fabs(acc);
            for (int32_t k = 0; k < K; ++k) {
                int64_t m = nmap[(size_t)k * (size_t)N + (size_t)n];
                if (m < 0 || m >= N) continue; /* sentinel or out of range: no term */
                for (int32_t ci = 0; ci < Ci; ++ci) {
                    double f = oracle_widen(feats, dtype, (size_t)m * (size_t)Ci + (size_t)ci);
                    double g = oracle_widen(w, dtype,
                                            ((size_t)k * (size_t)Ci + (size_t)ci) * (size_t)Co +
                                                (size_t)co);
                    double term = f * g;
                    acc += term;
                    mag += fabs(term);
                }
            }
            out[(size_t)r * (size_t)Co + (size_t)co] = acc;
            sabs[(size_t)r * (size_t)Co + (size_t)co] = mag;
        }
    }
    return ORACLE_OK;
}

/* Number of entries v of a (K, N) map with 0 <= v < N. */
int64_t oracle_count_valid_pairs(const int32_t* nmap, int64_t N, int32_t K)
{
    int64_t total = 0;
    for (size_t i = 0; i < (size_t)K * (size_t)N; ++i)
        if (nmap[i] >= 0 && nmap[i] < N) ++total;
    return total;
}

/*
 * Input gradient.  Computes the rows of dfeats listed in `rows` (all N rows
 * when rows == NULL): one pass over the whole map picks every valid entry
 * m = nmap[k, n] whose target m is listed and adds its terms
 * dout[n, co] * w[k, ci, co].  dabs receives sum |term|.
 */
int oracle_dgrad(const void* dout, int32_t dtype, const int32_t* nmap, const void* w, int64_t N,
                 int32_t K, int32_t Ci, int32_t Co, const int64_t* rows, int64_t n_rows,
                 double* out, double* dabs)
{
    if (N < 1 || K < 1 || Ci < 1 || Co < 1 || dout == NULL || nmap == NULL || w == NULL ||
        out == NULL || dabs == NULL)
        return ORACLE_ERR_INVALID_ARG;
    if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return ORACLE_ERR_INVALID_ARG;
    int64_t count = rows != NULL ? n_rows : N;
    int64_t* slot = (int64_t*)malloc((size_t)N * sizeof(int64_t));
    if (slot == NULL) return ORACLE_ERR_NOMEM;
    for (int64_t m = 0; m < N; ++m) slot[m] = rows != NULL ? -1 : m;
    if (rows != NULL) {
        for (int64_t r = 0; r < count; ++r) {
            if (rows[r] < 0 || rows[r] >= N) {
                free(slot);
                return ORACLE_ERR_INVALID_ARG;
            }
            slot[rows[r]] = r;
        }
    }
    memset(out, 0, (size_t)count * (size_t)Ci * sizeof(double));
    memset(dabs, 0, (size_t)count * (size_t)Ci * sizeof(double));
    for (int32_t k = 0; k < K; ++k) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t m = nmap[(size_t)k * (size_t)N + (size_t)n];
            if (m < 0 || m >= N || slot[m] < 0) continue;
            double* o = out + (size_t)slot[m] * (size_t)Ci;
            double* a = dabs + (size_t)slot[m] * (size_t)Ci;
            for (int32_t ci = 0; ci < Ci; ++ci) {
                double acc = 0.0, mag = 0.0;
                for (int32_t co = 0; co < Co; ++co) {
                    double g = oracle_widen(dout, dtype, (size_t)n * (size_t)Co + (size_t)co);
                    double v = oracle_widen(w, dtype,
                                            ((size_t)k * (size_t)Ci + (size_t)ci) * (size_t)Co +
                                                (size_t)co);
                    acc += g * v;
                    mag += fabs(g * v);
                }
                o[ci] += acc;
                a[ci] += mag;
            }
        }
    }
    free(slot);
    return ORACLE_OK;
}

/*
 * Weight gradient.  With entries == NULL computes all K * Ci * Co values of
 * dw (out laid out (K, Ci, Co)); otherwise the listed flat indices
 * (k * Ci + ci) * Co + co, one sum over all N voxels each.  dabs receives
 * sum |term|.
 */
int oracle_wgrad(const void* feats, const void* dout, int32_t dtype, const int32_t* nmap,
                 int64_t N, int32_t K, int32_t Ci, int32_t Co, const int64_t* entries,
                 int64_t n_entries, double* out, double* dabs)
{
    if (N < 1 || K < 1 || Ci < 1 || Co < 1 || feats == NULL || dout == NULL || nmap == NULL ||
        out == NULL || dabs == NULL)
        return ORACLE_ERR_INVALID_ARG;
    if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return ORACLE_ERR_INVALID_ARG;
    if (entries == NULL) {
        size_t total = (size_t)K * (size_t)Ci * (size_t)Co;
        memset(out, 0, total * sizeof(double));
        memset(dabs, 0, total * sizeof(double));
        for (int32_t k = 0; k < K; ++k) {
            for (int64_t n = 0; n < N; ++n) {
                int64_t m = nmap[(size_t)k * (size_t)N + (size_t)n];
                if (m < 0 || m >= N) continue;
                for (int32_t ci = 0; ci < Ci; ++ci) {
                    double f = oracle_widen(feats, dtype, (size_t)m * (size_t)Ci + (size_t)ci);
                    double* o = out + ((size_t)k * (size_t)Ci + (size_t)ci) * (size_t)Co;
                    double* a = dabs + ((size_t)k * (size_t)Ci + (size_t)ci) * (size_t)Co;
                    for (int32_t co = 0; co < Co; ++co) {
                        double t = f * oracle_widen(dout, dtype, (size_t)n * (size_t)Co + (size_t)co);
                        o[co] += t;
                        a[co] += fabs(t);
                    }
                }
            }
        }
        return ORACLE_OK;
    }
    for (int64_t e = 0; e < n_entries; ++e) {
        int64_t flat = entries[e];
        if (flat < 0 || flat >= (int64_t)K * Ci * Co) return ORACLE_ERR_INVALID_ARG;
        int32_t co = (int32_t)(flat % Co);
        int32_t ci = (int32_t)((flat / Co) % Ci);
        int32_t k = (int32_t)(flat / ((int64_t)Co * Ci));
        double acc = 0.0, mag = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            int64_t m = nmap[(size_t)k * (size_t)N + (size_t)n];
            if (m < 0 || m >= N) continue;
            double t = oracle_widen(feats, dtype, (size_t)m * (size_t)Ci + (size_t)ci) *
                       oracle_widen(dout, dtype, (size_t)n * (size_t)Co + (size_t)co);
            acc += t;
            mag += fabs(t);
        }
        out[e] = acc;
        dabs[e] = mag;
    }
    return ORACLE_OK;
}
