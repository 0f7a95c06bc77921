/*
 * pkv_c_consumer.c -- the C ABI of libpkv.so used from plain C, as a non-Python caller would
 * (test program; not part of the library).
 *
 * One layer of a two-layer fp16 cache with 8 query / 2 KV heads of 128 dims:
 *   1. the host block manager admits three prompts (37, 16 and 100 tokens) from a shuffled pool
 *      ("La idea de PagedAttention", steps 1-3: fixed blocks, a table per sequence, slots);
 *   2. pkv_kv_append writes their K/V rows into layer 1 of the device pools;
 *   3. one decode step: pkv_mgr_append_slot reserves each sequence's next slot, then
 *      pkv_paged_decode_append_attention appends the new rows and attends in one call (step 5);
 *   4. the result is compared with the fp64 oracle (oracle/oracle.c, test infrastructure) run on
 *      host copies of the same rows, written through the oracle's own append;
 *   5. the manager is saved and reloaded (pkv_mgr_save / pkv_mgr_load) and must carry on exactly
 *      like the original.
 * Exit status 0 and a line "c consumer ok" on success; the largest |gpu - oracle| must stay within
 * 2e-2 (fp16 inputs, fp32 accumulation), and the device status word must read 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "pkv.h"

/* from oracle/oracle.c (its own dtype codes: 1 = fp16) */
int oracle_kv_append(int elem_bytes, int n_kv, int head_dim, int block_size, int num_blocks, const void* k,
                     const void* v, const int64_t* slots, int n_tok, void* k_pool, void* v_pool);
int oracle_paged_decode(int dtype, int n_q, int n_kv, int head_dim, int block_size, int num_blocks, const void* q,
                        const void* k_pool, const void* v_pool, const int32_t* tables, int max_blocks,
                        const int32_t* lens, int n_seqs, double scale, double* out, int n_threads);
double oracle_elem_to_double(int dtype, const void* base, size_t i);

#define CHECK(x)                                                                   \
    do {                                                                           \
        if (!(x)) {                                                                \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #x);        \
            return 1;                                                              \
        }                                                                          \
    } while (0)
#define CUDA_OK(x) CHECK((x) == cudaSuccess)

/* fp32 -> fp16 bits, round to nearest even (values here are normal and small) */
static uint16_t to_half(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    const uint32_t sign = (x >> 16) & 0x8000u;
    int32_t e = (int32_t)((x >> 23) & 0xff) - 127 + 15;
    uint32_t m = x & 0x7fffffu;
    if (e <= 0) return (uint16_t)sign; /* flush tiny values (not produced here) */
    uint32_t h = ((uint32_t)e << 10) | (m >> 13);
    const uint32_t rest = m & 0x1fffu;
    if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) ++h;
    return (uint16_t)(sign | h);
}

static uint64_t rng_state = 0x9e3779b97f4a7c15ull;
static float uniform(void) { /* xorshift64*, in [-2, 2) */
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    const uint64_t r = rng_state * 0x2545f4914f6cdd1dull;
    return (float)((double)(r >> 11) / 9007199254740992.0 * 4.0 - 2.0);
}

int main(void) {
    const pkv_cache_desc desc = {PKV_F16, 2, 64, 8, 2, 128, 16};
    const int layer = 1, n_kv = 2, n_q = 8, d = 128, nb = 64, bs = 16, max_blocks = 8;
    CHECK(pkv_validate_desc(&desc) == PKV_OK);
    const size_t layer_elems = (size_t)nb * n_kv * bs * d;
    const size_t pool_bytes = (size_t)pkv_pool_bytes(&desc);
    CHECK(pool_bytes == 2 * layer_elems * 2);

    /* 1. admission from a shuffled free list */
    int32_t order[64];
    for (int i = 0; i < nb; ++i) order[i] = i;
    for (int i = nb - 1; i > 0; --i) {
        const int j = (int)((uniform() + 2.0f) / 4.0f * (float)(i + 1)) % (i + 1);
        const int32_t t = order[i];
        order[i] = order[j];
        order[j] = t;
    }
    pkv_mgr* mgr = pkv_mgr_create(nb, bs, order);
    CHECK(mgr != NULL);
    const int64_t ids[3] = {11, 12, 13};
    const int prompt[3] = {37, 16, 100};
    int n_tok = 0;
    int64_t slots[153];
    for (int s = 0; s < 3; ++s) {
        CHECK(pkv_mgr_add_seq(mgr, ids[s], prompt[s], 0, slots + n_tok) == PKV_OK);
        n_tok += prompt[s];
    }
    CHECK(n_tok == 153);

    /* 2. prompt rows -> layer 1 of the device pools */
    const size_t row = (size_t)n_kv * d;
    uint16_t* hk = malloc(sizeof(uint16_t) * n_tok * row);
    uint16_t* hv = malloc(sizeof(uint16_t) * n_tok * row);
    for (size_t i = 0; i < (size_t)n_tok * row; ++i) {
        hk[i] = to_half(uniform());
        hv[i] = to_half(uniform());
    }
    void *k_pool, *v_pool, *dk, *dv, *dslots;
    CUDA_OK(cudaMalloc(&k_pool, pool_bytes));
    CUDA_OK(cudaMalloc(&v_pool, pool_bytes));
    CUDA_OK(cudaMemset(k_pool, 0xff, pool_bytes)); /* NaN everywhere no row was written */
    CUDA_OK(cudaMemset(v_pool, 0xff, pool_bytes));
    CUDA_OK(cudaMalloc(&dk, sizeof(uint16_t) * n_tok * row));
    CUDA_OK(cudaMalloc(&dv, sizeof(uint16_t) * n_tok * row));
    CUDA_OK(cudaMalloc(&dslots, sizeof(int64_t) * n_tok));
    CUDA_OK(cudaMemcpy(dk, hk, sizeof(uint16_t) * n_tok * row, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dv, hv, sizeof(uint16_t) * n_tok * row, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dslots, slots, sizeof(int64_t) * n_tok, cudaMemcpyHostToDevice));
    CHECK(pkv_kv_append(&desc, layer, dk, dv, (const int64_t*)dslots, n_tok, k_pool, v_pool, NULL) == PKV_OK);

    /* 3. one decode step: reserve the next slot of every sequence, then append + attend */
    int64_t new_slot[3];
    for (int s = 0; s < 3; ++s) {
        int32_t src = -2, dst = -2;
        CHECK(pkv_mgr_append_slot(mgr, ids[s], &new_slot[s], &src, &dst) == PKV_OK);
        CHECK(src == -1 && dst == -1); /* nothing is shared: no copy-on-write */
    }
    int32_t tables[3 * 8], lens[3];
    CHECK(pkv_mgr_pack_tables(mgr, ids, 3, max_blocks, tables, lens) == PKV_OK);
    for (int s = 0; s < 3; ++s) CHECK(lens[s] == prompt[s] + 1);
    uint16_t hq[3 * 8 * 128], hkn[3 * 2 * 128], hvn[3 * 2 * 128];
    for (int i = 0; i < 3 * n_q * d; ++i) hq[i] = to_half(uniform());
    for (int i = 0; i < 3 * n_kv * d; ++i) {
        hkn[i] = to_half(uniform());
        hvn[i] = to_half(uniform());
    }
    void *dq, *dkn, *dvn, *dmeta, *dout, *ws = NULL;
    CUDA_OK(cudaMalloc(&dq, sizeof hq));
    CUDA_OK(cudaMalloc(&dkn, sizeof hkn));
    CUDA_OK(cudaMalloc(&dvn, sizeof hvn));
    CUDA_OK(cudaMalloc(&dmeta, sizeof tables + sizeof lens));
    CUDA_OK(cudaMalloc(&dout, sizeof hq));
    CUDA_OK(cudaMemcpy(dq, hq, sizeof hq, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dkn, hkn, sizeof hkn, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dvn, hvn, sizeof hvn, cudaMemcpyHostToDevice));
    /* the step's tables and lengths as one pinned image (27 words: six 16-byte words and a
     * 4-byte tail), uploaded by pkv_upload_metadata; pageable memory is refused */
    int32_t* hmeta = NULL;
    CUDA_OK(cudaMallocHost((void**)&hmeta, sizeof tables + sizeof lens));
    memcpy(hmeta, tables, sizeof tables);
    memcpy(hmeta + 3 * 8, lens, sizeof lens);
    CHECK(pkv_upload_metadata(dmeta, tables, sizeof tables, NULL) == PKV_ERR_INVALID_ARG);
    CHECK(pkv_upload_metadata(dmeta, hmeta, sizeof tables + sizeof lens, NULL) == PKV_OK);
    const int32_t* dtab = (const int32_t*)dmeta;
    const int32_t* dlens = (const int32_t*)dmeta + 3 * 8;
    const size_t ws_bytes = pkv_decode_workspace_bytes(&desc, 3, max_blocks);
    if (ws_bytes) CUDA_OK(cudaMalloc(&ws, ws_bytes));
    const float scale = 1.0f / sqrtf((float)d);
    CHECK(pkv_paged_decode_append_attention(&desc, layer, dq, dkn, dvn, k_pool, v_pool, dtab, max_blocks, dlens, 3,
                                            scale, dout, ws, ws_bytes, NULL) == PKV_OK);
    CUDA_OK(cudaDeviceSynchronize());
    {
        int32_t back[3 * 8 + 3];
        CUDA_OK(cudaMemcpy(back, dmeta, sizeof back, cudaMemcpyDeviceToHost));
        CHECK(memcmp(back, hmeta, sizeof back) == 0);
    }
    uint32_t flags = 1;
    CHECK(pkv_get_device_status(NULL, &flags) == PKV_OK && flags == 0);
    uint16_t hout[3 * 8 * 128];
    CUDA_OK(cudaMemcpy(hout, dout, sizeof hout, cudaMemcpyDeviceToHost));

    /* 4. the oracle on host copies: its own append of the same rows, then fp64 attention */
    uint16_t* ok_pool = malloc(sizeof(uint16_t) * layer_elems);
    uint16_t* ov_pool = malloc(sizeof(uint16_t) * layer_elems);
    memset(ok_pool, 0, sizeof(uint16_t) * layer_elems);
    memset(ov_pool, 0, sizeof(uint16_t) * layer_elems);
    CHECK(oracle_kv_append(2, n_kv, d, bs, nb, hk, hv, slots, n_tok, ok_pool, ov_pool) == 0);
    CHECK(oracle_kv_append(2, n_kv, d, bs, nb, hkn, hvn, new_slot, 3, ok_pool, ov_pool) == 0);
    double ref[3 * 8 * 128];
    CHECK(oracle_paged_decode(1, n_q, n_kv, d, bs, nb, hq, ok_pool, ov_pool, tables, max_blocks, lens, 3,
                              (double)scale, ref, 1) == 0);
    double err = 0.0;
    for (int i = 0; i < 3 * n_q * d; ++i) {
        const double e = fabs(oracle_elem_to_double(1, hout, (size_t)i) - ref[i]);
        if (!(e <= err)) err = e; /* NaN propagates into err */
    }
    /* the device pools hold exactly the oracle's rows at every written slot (bit-exact append) */
    uint16_t* dev_layer = malloc(sizeof(uint16_t) * layer_elems);
    for (int kv = 0; kv < 2; ++kv) {
        CUDA_OK(cudaMemcpy(dev_layer, (char*)(kv ? v_pool : k_pool) + layer_elems * 2, sizeof(uint16_t) * layer_elems,
                           cudaMemcpyDeviceToHost));
        const uint16_t* want = kv ? ov_pool : ok_pool;
        for (int t = 0; t < n_tok + 3; ++t) {
            const int64_t sl = t < n_tok ? slots[t] : new_slot[t - n_tok];
            for (int g = 0; g < n_kv; ++g) {
                const size_t off = (((size_t)(sl / bs) * n_kv + g) * bs + (size_t)(sl % bs)) * d;
                CHECK(memcmp(dev_layer + off, want + off, sizeof(uint16_t) * d) == 0);
            }
        }
    }
    /* 5. checkpoint / resume: a manager reloaded from its saved image packs the same tables and
     *    hands out the same next slots as the original */
    const size_t img_bytes = pkv_mgr_save_bytes(mgr);
    unsigned char* img = malloc(img_bytes);
    size_t written = 0;
    CHECK(img != NULL && pkv_mgr_save(mgr, img, img_bytes, &written) == PKV_OK && written == img_bytes);
    pkv_mgr* again = pkv_mgr_load(img, written);
    CHECK(again != NULL);
    int32_t tables2[3 * 8], lens2[3];
    CHECK(pkv_mgr_pack_tables(again, ids, 3, max_blocks, tables2, lens2) == PKV_OK);
    CHECK(memcmp(tables, tables2, sizeof tables) == 0 && memcmp(lens, lens2, sizeof lens) == 0);
    for (int s = 0; s < 3; ++s) {
        int64_t a = -1, b = -2;
        int32_t s1, d1, s2, d2;
        CHECK(pkv_mgr_append_slot(mgr, ids[s], &a, &s1, &d1) == PKV_OK);
        CHECK(pkv_mgr_append_slot(again, ids[s], &b, &s2, &d2) == PKV_OK);
        CHECK(a == b && s1 == s2 && d1 == d2);
    }
    img[written / 2] ^= 1u; /* a corrupted image is refused */
    CHECK(pkv_mgr_load(img, written) == NULL);
    free(img);
    pkv_mgr_destroy(again);

    printf("c consumer ok: max |gpu - oracle| = %.3g over %d outputs\n", err, 3 * n_q * d);
    CHECK(err <= 2e-2);
    pkv_mgr_destroy(mgr);
    return 0;
}
