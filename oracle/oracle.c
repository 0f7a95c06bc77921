/*
 * oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, fp64 CPU restatement of what the paged KV cache hot path computes.
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg may
 * load it. It shares no code, header, table or helper with the CUDA library: it has its
 * own dtype codes, its own bit-level fp16/bf16 decoders and its own pool indexing.
 *
 * What it restates (sources are the three pages on paged KV caches):
 *  - "04 - Hacia PagedAttention (vista previa)", section "La idea de PagedAttention":
 *      step 1  the KV cache is cut into fixed blocks of B_block tokens;
 *      step 2  a per-sequence block table maps logical block i to physical block X;
 *      step 3  appending a token writes into the last block (slot = X*B_block + offset);
 *      step 5  attention takes the block table and gathers the rows itself (decode: one
 *              query per sequence; prefill: a chunk of causal queries per sequence).
 *    Section "Lo que deberias llevarte", item 2: paging changes the memory layout only, so
 *    the result is exactly dense softmax attention over the gathered rows.
 *  - "PagedAttention e continuous batching", section "01 - Conceito", paragraph 6:
 *    copy-on-write gives the diverging branch a fresh copy of the shared block.
 *  - "Paged Attention em Large Language Models LLMs", section "Configurando as
 *    Constantes": KV bytes per token = 2 * layers * heads * head_dim * bytes.
 *
 * Readings taken where the pages are silent (each one is listed in the design notes):
 *  - pool layout per layer is [num_blocks][n_kv][block_size][head_dim], row-major;
 *  - query head h reads KV head h / (n_q / n_kv) (consecutive query heads share one);
 *  - a sequence with context length 0 attends to nothing and outputs zeros.
 *
 * Arithmetic: every element is widened exactly to double, logits are
 * z_j = scale * sum_i q_i k_ji, the softmax subtracts the maximum logit and uses libm exp,
 * and the output is sum_j (w_j / Z) v_j -- the textbook definition, in that order.
 * OpenMP only distributes independent (sequence, head) pairs; it never changes the
 * arithmetic of one pair.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* The oracle's own element type codes. */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

static size_t orc_elem_bytes(int dtype) {
    switch (dtype) {
    case ORC_F32: return 4;
    case ORC_F16: return 2;
    case ORC_BF16: return 2;
    default: return 0;
    }
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double orc_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/2^10) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
static double orc_bf16_to_double(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133); /* subnormal: f * 2^-126 * 2^-7 */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + f), e - 134); /* (1 + f/2^7) * 2^(e-127) */
    }
    return sign ? -v : v;
}

static double orc_load(int dtype, const void* base, size_t i) {
    if (dtype == ORC_F32) {
        float x;
        memcpy(&x, (const char*)base + 4 * i, 4);
        return (double)x;
    }
    uint16_t u;
    memcpy(&u, (const char*)base + 2 * i, 2);
    return dtype == ORC_F16 ? orc_half_to_double(u) : orc_bf16_to_double(u);
}

/* Exposed so tests can check the decoders against an independent library conversion. */
double oracle_elem_to_double(int dtype, const void* base, size_t i) {
    return orc_load(dtype, base, i);
}

/* Bulk form of the above, for exhaustive decoder checks. */
void oracle_elems_to_double(int dtype, const void* base, size_t n, double* out) {
    for (size_t i = 0; i < n; ++i) out[i] = orc_load(dtype, base, i);
}

/* "Configurando as Constantes": 2 (K and V) * layers * kv heads * head_dim * bytes. */
uint64_t oracle_kv_bytes_per_token(int n_layers, int n_kv_heads, int head_dim, int elem_bytes) {
    return 2ull * (uint64_t)n_layers * (uint64_t)n_kv_heads * (uint64_t)head_dim * (uint64_t)elem_bytes;
}

/* Flat index of row (physical block, kv head, offset) in one layer's pool. */
static size_t orc_row(int64_t phys, int g, int off, int n_kv, int block_size, int head_dim) {
    return (((size_t)phys * (size_t)n_kv + (size_t)g) * (size_t)block_size + (size_t)off) * (size_t)head_dim;
}

/*
 * Paged decode attention for one layer, one query token per sequence.
 *   q        [n_seqs][n_q][head_dim]                    (dtype)
 *   k_pool   [num_blocks][n_kv][block_size][head_dim]   (dtype)
 *   v_pool   same layout as k_pool
 *   tables   [n_seqs][max_blocks] int32, logical block -> physical block
 *   lens     [n_seqs] int32 context lengths (including the newest token)
 *   out      [n_seqs][n_q][head_dim] double
 * Returns 0, or -1 if an argument is malformed (the oracle refuses instead of guessing):
 * a table entry outside [0, num_blocks), a length outside [0, max_blocks*block_size],
 * or n_q not a multiple of n_kv.
 */
int oracle_paged_decode(int dtype, int n_q, int n_kv, int head_dim, int block_size, int num_blocks,
                        const void* q, const void* k_pool, const void* v_pool,
                        const int32_t* tables, int max_blocks, const int32_t* lens, int n_seqs,
                        double scale, double* out, int n_threads) {
    if (orc_elem_bytes(dtype) == 0 || n_q <= 0 || n_kv <= 0 || n_q % n_kv != 0 || head_dim <= 0 ||
        block_size <= 0 || n_seqs < 0)
        return -1;
    const int group = n_q / n_kv;
    for (int s = 0; s < n_seqs; ++s) {
        if (lens[s] < 0 || (int64_t)lens[s] > (int64_t)max_blocks * block_size) return -1;
        int nb = (lens[s] + block_size - 1) / block_size;
        for (int i = 0; i < nb; ++i) {
            int32_t x = tables[(size_t)s * max_blocks + i];
            if (x < 0 || x >= num_blocks) return -1;
        }
    }
    if (n_threads < 1) n_threads = 1;
    const long n_pairs = (long)n_seqs * n_q;
    int failed = 0;

#pragma omp parallel for num_threads(n_threads) schedule(dynamic, 1)
    for (long sh = 0; sh < n_pairs; ++sh) {
        const int s = (int)(sh / n_q);
        const int h = (int)(sh % n_q);
        const int g = h / group;
        const int n = lens[s];
        double* o = out + ((size_t)s * n_q + h) * head_dim;
        if (n == 0) {
            for (int i = 0; i < head_dim; ++i) o[i] = 0.0;
            continue;
        }
        double* kc = (double*)malloc(sizeof(double) * (size_t)n * head_dim);
        double* vc = (double*)malloc(sizeof(double) * (size_t)n * head_dim);
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        double* z = (double*)malloc(sizeof(double) * (size_t)n);
        if (!kc || !vc || !qv || !z) {
            free(kc); free(vc); free(qv); free(z);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        /* Step 5 of "La idea de PagedAttention": follow the table, gather the logical rows. */
        for (int j = 0; j < n; ++j) {
            int64_t phys = tables[(size_t)s * max_blocks + j / block_size];
            size_t row = orc_row(phys, g, j % block_size, n_kv, block_size, head_dim);
            for (int i = 0; i < head_dim; ++i) {
                kc[(size_t)j * head_dim + i] = orc_load(dtype, k_pool, row + i);
                vc[(size_t)j * head_dim + i] = orc_load(dtype, v_pool, row + i);
            }
        }
        for (int i = 0; i < head_dim; ++i) qv[i] = orc_load(dtype, q, ((size_t)s * n_q + h) * head_dim + i);
        /* Dense softmax attention over the gathered rows. */
        double m = -INFINITY;
        for (int j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int i = 0; i < head_dim; ++i) acc += qv[i] * kc[(size_t)j * head_dim + i];
            z[j] = scale * acc;
            if (z[j] > m) m = z[j];
        }
        double zsum = 0.0;
        for (int j = 0; j < n; ++j) {
            z[j] = exp(z[j] - m);
            zsum += z[j];
        }
        for (int i = 0; i < head_dim; ++i) {
            double acc = 0.0;
            for (int j = 0; j < n; ++j) acc += (z[j] / zsum) * vc[(size_t)j * head_dim + i];
            o[i] = acc;
        }
        free(kc); free(vc); free(qv); free(z);
    }
    return failed ? -1 : 0;
}

/*
 * Paged prefill attention for one layer: a chunk of several new query tokens per sequence,
 * each attending causally to the sequence's cache through its block table.
 * "PagedAttention e continuous batching", section "01 - Conceito", paragraph 5 slices a long
 * prompt into chunks that share steps with decoding; "La idea de PagedAttention", step 5, has
 * the kernel gather the rows through the table. Reading taken (the pages give no formula for
 * the chunk): the n_s tokens of sequence s's chunk are its newest, already appended, so with
 * c = lens[s] they sit at positions c - n_s .. c - 1, and the token at position p attends to
 * positions 0 .. p (causal), exactly as dense causal attention over the gathered rows.
 *   q            [n_tokens][n_q][head_dim] (dtype); the tokens of sequence s are rows
 *                query_start[s] .. query_start[s+1]-1, in position order
 *   query_start  [n_seqs + 1] int32, non-decreasing, query_start[0] >= 0,
 *                query_start[n_seqs] <= n_tokens
 *   lens         [n_seqs] int32 context lengths after the chunk (>= the chunk's length)
 *   out          [n_tokens][n_q][head_dim] double; rows of no sequence are left untouched
 * Returns 0, or -1 on malformed arguments (as oracle_paged_decode, plus a chunk longer than its
 * context or a query_start out of order or out of range).
 */
int oracle_paged_prefill(int dtype, int n_q, int n_kv, int head_dim, int block_size, int num_blocks,
                         const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* tables, int max_blocks, const int32_t* lens,
                         const int32_t* query_start, int n_seqs, int n_tokens,
                         double scale, double* out, int n_threads) {
    if (orc_elem_bytes(dtype) == 0 || n_q <= 0 || n_kv <= 0 || n_q % n_kv != 0 || head_dim <= 0 ||
        block_size <= 0 || n_seqs < 0 || n_tokens < 0)
        return -1;
    if (n_seqs > 0 && (query_start[0] < 0 || query_start[n_seqs] > n_tokens)) return -1;
    const int group = n_q / n_kv;
    for (int s = 0; s < n_seqs; ++s) {
        const int n_new = query_start[s + 1] - query_start[s];
        if (n_new < 0 || lens[s] < n_new || (int64_t)lens[s] > (int64_t)max_blocks * block_size) return -1;
        int nb = (lens[s] + block_size - 1) / block_size;
        for (int i = 0; i < nb; ++i) {
            int32_t x = tables[(size_t)s * max_blocks + i];
            if (x < 0 || x >= num_blocks) return -1;
        }
    }
    if (n_threads < 1) n_threads = 1;
    const long n_pairs = (long)n_seqs * n_q;
    int failed = 0;

#pragma omp parallel for num_threads(n_threads) schedule(dynamic, 1)
    for (long sh = 0; sh < n_pairs; ++sh) {
        const int s = (int)(sh / n_q);
        const int h = (int)(sh % n_q);
        const int g = h / group;
        const int c = lens[s];
        const int n_new = query_start[s + 1] - query_start[s];
        if (n_new == 0) continue;
        double* kc = (double*)malloc(sizeof(double) * (size_t)c * head_dim);
        double* vc = (double*)malloc(sizeof(double) * (size_t)c * head_dim);
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        double* z = (double*)malloc(sizeof(double) * (size_t)c);
        if (!kc || !vc || !qv || !z) {
            free(kc); free(vc); free(qv); free(z);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        /* Gather the sequence's logical rows through its table, once per (sequence, head). */
        for (int j = 0; j < c; ++j) {
            int64_t phys = tables[(size_t)s * max_blocks + j / block_size];
            size_t row = orc_row(phys, g, j % block_size, n_kv, block_size, head_dim);
            for (int i = 0; i < head_dim; ++i) {
                kc[(size_t)j * head_dim + i] = orc_load(dtype, k_pool, row + i);
                vc[(size_t)j * head_dim + i] = orc_load(dtype, v_pool, row + i);
            }
        }
        for (int t = 0; t < n_new; ++t) {
            const size_t qrow = ((size_t)(query_start[s] + t) * n_q + h) * head_dim;
            const int pos = c - n_new + t; /* this query's position: it sees keys 0 .. pos */
            for (int i = 0; i < head_dim; ++i) qv[i] = orc_load(dtype, q, qrow + i);
            double m = -INFINITY;
            for (int j = 0; j <= pos; ++j) {
                double acc = 0.0;
                for (int i = 0; i < head_dim; ++i) acc += qv[i] * kc[(size_t)j * head_dim + i];
                z[j] = scale * acc;
                if (z[j] > m) m = z[j];
            }
            double zsum = 0.0;
            for (int j = 0; j <= pos; ++j) {
                z[j] = exp(z[j] - m);
                zsum += z[j];
            }
            double* o = out + qrow;
            for (int i = 0; i < head_dim; ++i) {
                double acc = 0.0;
                for (int j = 0; j <= pos; ++j) acc += (z[j] / zsum) * vc[(size_t)j * head_dim + i];
                o[i] = acc;
            }
        }
        free(kc); free(vc); free(qv); free(z);
    }
    return failed ? -1 : 0;
}

/*
 * KV append for one layer ("La idea de PagedAttention", step 3): token t's K and V rows for
 * every kv head go to row (slot / block_size, head, slot % block_size) of the pools.
 * A negative slot marks a padding token and is skipped. Pure byte copies.
 *   k, v  [n_tok][n_kv][head_dim] elements of elem_bytes each
 * Returns 0, or -1 if a slot lies beyond the pool.
 */
int oracle_kv_append(int elem_bytes, int n_kv, int head_dim, int block_size, int num_blocks,
                     const void* k, const void* v, const int64_t* slots, int n_tok,
                     void* k_pool, void* v_pool) {
    const size_t row_bytes = (size_t)head_dim * (size_t)elem_bytes;
    for (int t = 0; t < n_tok; ++t) {
        if (slots[t] >= (int64_t)num_blocks * block_size) return -1;
    }
    for (int t = 0; t < n_tok; ++t) {
        int64_t slot = slots[t];
        if (slot < 0) continue;
        int64_t phys = slot / block_size;
        int off = (int)(slot % block_size);
        for (int g = 0; g < n_kv; ++g) {
            size_t dst = orc_row(phys, g, off, n_kv, block_size, head_dim) * (size_t)elem_bytes;
            size_t src = ((size_t)t * n_kv + g) * row_bytes;
            memcpy((char*)k_pool + dst, (const char*)k + src, row_bytes);
            memcpy((char*)v_pool + dst, (const char*)v + src, row_bytes);
        }
    }
    return 0;
}

/*
 * Copy-on-write block copy ("01 - Conceito", paragraph 6): for every (src, dst) pair, the
 * whole physical block src -- all layers, all kv heads, all offsets, K and V -- is copied
 * to dst. pools are [n_layers][num_blocks][n_kv][block_size][head_dim].
 * Returns 0, or -1 if an id lies outside [0, num_blocks).
 */
int oracle_copy_blocks(int elem_bytes, int n_layers, int n_kv, int head_dim, int block_size, int num_blocks,
                       void* k_pool, void* v_pool, const int32_t* pairs, int n_pairs) {
    for (int i = 0; i < 2 * n_pairs; ++i) {
        if (pairs[i] < 0 || pairs[i] >= num_blocks) return -1;
    }
    const size_t block_bytes = (size_t)n_kv * block_size * head_dim * elem_bytes;
    const size_t layer_bytes = block_bytes * (size_t)num_blocks;
    for (int p = 0; p < n_pairs; ++p) {
        size_t src = (size_t)pairs[2 * p] * block_bytes;
        size_t dst = (size_t)pairs[2 * p + 1] * block_bytes;
        for (int l = 0; l < n_layers; ++l) {
            memcpy((char*)k_pool + l * layer_bytes + dst, (const char*)k_pool + l * layer_bytes + src, block_bytes);
            memcpy((char*)v_pool + l * layer_bytes + dst, (const char*)v_pool + l * layer_bytes + src, block_bytes);
        }
    }
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
