/*
 * manager.c -- host block manager of the paged KV cache (pure C11, no CUDA).
 *
 * Implements the bookkeeping of "04 - Hacia PagedAttention (vista previa)", section
 * "La idea de PagedAttention" (steps 1-4: fixed blocks, per-sequence block tables, append
 * into the last block or a fresh one, free to a free list) and of "PagedAttention e
 * continuous batching", section "01 - Conceito" (paragraph 6: shared prefix blocks,
 * copy-on-write, reference counts; paragraph 7: admission in countable blocks that refuses
 * early; paragraph 8: block metrics).
 *
 * Data structures:
 *   free list  ring buffer of num_blocks ids (FIFO: pop front, push back; rollback pushes
 *              front, which restores the exact previous order);
 *   refcounts  int32 per physical block;
 *   sequences  open-addressing hash map (linear probing, backward-shift deletion) from the
 *              caller's int64 id to {table, n_blocks, capacity, context length}.
 * Every operation checks everything and reserves any host memory it needs before it
 * changes state, so a failed operation leaves the state unchanged.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "pkv.h"

typedef struct {
    int64_t id;
    int32_t* table;
    int32_t n_blocks;
    int32_t cap;
    int32_t ctx;
    int32_t used; /* slot occupied */
} seq_rec;

struct pkv_mgr {
    int32_t num_blocks;
    int32_t block_size;
    int32_t* ring; /* free list storage, capacity num_blocks */
    int32_t head;
    int32_t n_free;
    int32_t* ref;
    seq_rec* map;
    int64_t map_cap; /* power of two */
    int64_t n_seqs;
    int64_t alloc_failures;
    int64_t prefix_hits;
    int64_t cow_copies;
    int64_t append_oom;
    int32_t inject_after; /* < 0: disabled */
};

/* ---- sequence map ---------------------------------------------------------------------- */

static uint64_t mix64(uint64_t x) { /* splitmix64 finaliser */
    x ^= x >> 30;
    x *= 0xbf58476d1ce4e5b9ull;
    x ^= x >> 27;
    x *= 0x94d049bb133111ebull;
    x ^= x >> 31;
    return x;
}

static int64_t map_find(const pkv_mgr* m, int64_t id) {
    const uint64_t mask = (uint64_t)m->map_cap - 1;
    for (uint64_t i = mix64((uint64_t)id) & mask;; i = (i + 1) & mask) {
        if (!m->map[i].used) return -1;
        if (m->map[i].id == id) return (int64_t)i;
    }
}

static int map_grow(pkv_mgr* m) {
    int64_t ncap = m->map_cap * 2;
    seq_rec* nm = (seq_rec*)calloc((size_t)ncap, sizeof(seq_rec));
    if (!nm) return 0;
    const uint64_t mask = (uint64_t)ncap - 1;
    for (int64_t i = 0; i < m->map_cap; ++i) {
        if (!m->map[i].used) continue;
        uint64_t j = mix64((uint64_t)m->map[i].id) & mask;
        while (nm[j].used) j = (j + 1) & mask;
        nm[j] = m->map[i];
    }
    free(m->map);
    m->map = nm;
    m->map_cap = ncap;
    return 1;
}

/* Make room for one more sequence (keeps the load factor <= 1/2). */
static int map_reserve_one(pkv_mgr* m) {
    if ((m->n_seqs + 1) * 2 <= m->map_cap) return 1;
    return map_grow(m);
}

static seq_rec* map_insert(pkv_mgr* m, int64_t id) { /* caller reserved room, id is new */
    const uint64_t mask = (uint64_t)m->map_cap - 1;
    uint64_t i = mix64((uint64_t)id) & mask;
    while (m->map[i].used) i = (i + 1) & mask;
    memset(&m->map[i], 0, sizeof(seq_rec));
    m->map[i].id = id;
    m->map[i].used = 1;
    m->n_seqs++;
    return &m->map[i];
}

static void map_erase(pkv_mgr* m, int64_t pos) { /* backward-shift deletion */
    const uint64_t mask = (uint64_t)m->map_cap - 1;
    uint64_t hole = (uint64_t)pos;
    m->map[hole].used = 0;
    for (uint64_t i = (hole + 1) & mask; m->map[i].used; i = (i + 1) & mask) {
        uint64_t home = mix64((uint64_t)m->map[i].id) & mask;
        /* move i into the hole if its home is not in (hole, i] cyclically */
        int in_range = (hole <= i) ? (home > hole && home <= i) : (home > hole || home <= i);
        if (!in_range) {
            m->map[hole] = m->map[i];
            m->map[i].used = 0;
            hole = i;
        }
    }
    m->n_seqs--;
}

/* ---- free list ------------------------------------------------------------------------- */

static int32_t ring_pop_front(pkv_mgr* m) {
    int32_t b = m->ring[m->head];
    m->head = (m->head + 1) % m->num_blocks;
    m->n_free--;
    return b;
}

static void ring_push_back(pkv_mgr* m, int32_t b) {
    m->ring[(m->head + m->n_free) % m->num_blocks] = b;
    m->n_free++;
}

static void ring_push_front(pkv_mgr* m, int32_t b) {
    m->head = (m->head + m->num_blocks - 1) % m->num_blocks;
    m->ring[m->head] = b;
    m->n_free++;
}

/* Take one block (refcount 1). Returns -1 when the pool is empty or a failure is injected. */
static int32_t alloc_one(pkv_mgr* m) {
    if (m->inject_after == 0) {
        m->inject_after = -1;
        return -1;
    }
    if (m->inject_after > 0) m->inject_after--;
    if (m->n_free == 0) return -1;
    int32_t b = ring_pop_front(m);
    m->ref[b] = 1;
    return b;
}

static int ensure_table_cap(seq_rec* s, int32_t need) {
    if (need <= s->cap) return 1;
    int32_t ncap = s->cap ? s->cap : 4;
    while (ncap < need) ncap *= 2;
    int32_t* nt = (int32_t*)realloc(s->table, sizeof(int32_t) * (size_t)ncap);
    if (!nt) return 0;
    s->table = nt;
    s->cap = ncap;
    return 1;
}

static int32_t blocks_for(const pkv_mgr* m, int64_t tokens) {
    return (int32_t)((tokens + m->block_size - 1) / m->block_size);
}

/* ---- public API ------------------------------------------------------------------------ */

pkv_mgr* pkv_mgr_create(int32_t num_blocks, int32_t block_size, const int32_t* initial_free_order) {
    if (num_blocks <= 0 || block_size <= 0) return NULL;
    pkv_mgr* m = (pkv_mgr*)calloc(1, sizeof(pkv_mgr));
    if (!m) return NULL;
    m->num_blocks = num_blocks;
    m->block_size = block_size;
    m->ring = (int32_t*)malloc(sizeof(int32_t) * (size_t)num_blocks);
    m->ref = (int32_t*)calloc((size_t)num_blocks, sizeof(int32_t));
    m->map_cap = 64;
    m->map = (seq_rec*)calloc((size_t)m->map_cap, sizeof(seq_rec));
    if (!m->ring || !m->ref || !m->map) {
        pkv_mgr_destroy(m);
        return NULL;
    }
    if (initial_free_order) {
        /* must be a permutation of 0..num_blocks-1 */
        for (int32_t i = 0; i < num_blocks; ++i) {
            int32_t b = initial_free_order[i];
            if (b < 0 || b >= num_blocks || m->ref[b]) {
                pkv_mgr_destroy(m);
                return NULL;
            }
            m->ref[b] = 1; /* temporary "seen" mark */
            m->ring[i] = b;
        }
        memset(m->ref, 0, sizeof(int32_t) * (size_t)num_blocks);
    } else {
        for (int32_t i = 0; i < num_blocks; ++i) m->ring[i] = i;
    }
    m->head = 0;
    m->n_free = num_blocks;
    m->inject_after = -1;
    return m;
}

void pkv_mgr_destroy(pkv_mgr* m) {
    if (!m) return;
    if (m->map) {
        for (int64_t i = 0; i < m->map_cap; ++i)
            if (m->map[i].used) free(m->map[i].table);
        free(m->map);
    }
    free(m->ring);
    free(m->ref);
    free(m);
}

pkv_mgr* pkv_mgr_clone(const pkv_mgr* src) {
    if (!src) return NULL;
    pkv_mgr* m = (pkv_mgr*)calloc(1, sizeof(pkv_mgr));
    if (!m) return NULL;
    *m = *src;
    m->ring = (int32_t*)malloc(sizeof(int32_t) * (size_t)src->num_blocks);
    m->ref = (int32_t*)malloc(sizeof(int32_t) * (size_t)src->num_blocks);
    m->map = (seq_rec*)calloc((size_t)src->map_cap, sizeof(seq_rec));
    if (!m->ring || !m->ref || !m->map) {
        free(m->ring); free(m->ref); free(m->map); free(m);
        return NULL;
    }
    memcpy(m->ring, src->ring, sizeof(int32_t) * (size_t)src->num_blocks);
    memcpy(m->ref, src->ref, sizeof(int32_t) * (size_t)src->num_blocks);
    for (int64_t i = 0; i < src->map_cap; ++i) {
        if (!src->map[i].used) continue;
        m->map[i] = src->map[i];
        m->map[i].table = NULL;
        if (src->map[i].cap > 0) {
            m->map[i].table = (int32_t*)malloc(sizeof(int32_t) * (size_t)src->map[i].cap);
            if (!m->map[i].table) {
                pkv_mgr_destroy(m);
                return NULL;
            }
            memcpy(m->map[i].table, src->map[i].table, sizeof(int32_t) * (size_t)src->map[i].n_blocks);
        }
    }
    return m;
}

int pkv_mgr_add_seq(pkv_mgr* m, int64_t seq_id, int32_t n_prompt, int32_t reserve_tokens, int64_t* slots_out) {
    if (!m || n_prompt < 0 || reserve_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (map_find(m, seq_id) >= 0) return PKV_ERR_INVALID_ARG;
    const int32_t need = blocks_for(m, n_prompt);
    if ((int64_t)need + blocks_for(m, reserve_tokens) > m->n_free) {
        m->alloc_failures++;
        return PKV_ERR_NO_BLOCKS;
    }
    int32_t* table = NULL;
    if (need > 0) {
        table = (int32_t*)malloc(sizeof(int32_t) * (size_t)need);
        if (!table) return PKV_ERR_BAD_STATE;
    }
    if (!map_reserve_one(m)) {
        free(table);
        return PKV_ERR_BAD_STATE;
    }
    for (int32_t i = 0; i < need; ++i) {
        int32_t b = alloc_one(m);
        if (b < 0) { /* injected failure: undo in reverse so the free list is restored exactly */
            for (int32_t k = i - 1; k >= 0; --k) {
                m->ref[table[k]] = 0;
                ring_push_front(m, table[k]);
            }
            free(table);
            m->alloc_failures++;
            return PKV_ERR_NO_BLOCKS;
        }
        table[i] = b;
    }
    seq_rec* s = map_insert(m, seq_id);
    s->table = table;
    s->n_blocks = need;
    s->cap = need;
    s->ctx = n_prompt;
    if (slots_out) {
        for (int32_t p = 0; p < n_prompt; ++p)
            slots_out[p] = (int64_t)table[p / m->block_size] * m->block_size + p % m->block_size;
    }
    return PKV_OK;
}

int pkv_mgr_fork(pkv_mgr* m, int64_t parent, int64_t child) {
    if (!m || parent == child) return PKV_ERR_INVALID_ARG;
    if (map_find(m, child) >= 0) return PKV_ERR_INVALID_ARG;
    int64_t pp = map_find(m, parent);
    if (pp < 0) return PKV_ERR_INVALID_ARG;
    const int32_t nb = m->map[pp].n_blocks;
    int32_t* table = NULL;
    if (nb > 0) {
        table = (int32_t*)malloc(sizeof(int32_t) * (size_t)nb);
        if (!table) return PKV_ERR_BAD_STATE;
        memcpy(table, m->map[pp].table, sizeof(int32_t) * (size_t)nb);
    }
    const int32_t ctx = m->map[pp].ctx;
    if (!map_reserve_one(m)) { /* may move records: parent index is not used after this */
        free(table);
        return PKV_ERR_BAD_STATE;
    }
    for (int32_t i = 0; i < nb; ++i) m->ref[table[i]]++;
    seq_rec* s = map_insert(m, child);
    s->table = table;
    s->n_blocks = nb;
    s->cap = nb;
    s->ctx = ctx;
    m->prefix_hits += nb;
    return PKV_OK;
}

int pkv_mgr_append_slot(pkv_mgr* m, int64_t seq_id, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
    if (!m || !slot) return PKV_ERR_INVALID_ARG;
    int64_t pos = map_find(m, seq_id);
    if (pos < 0) return PKV_ERR_INVALID_ARG;
    seq_rec* s = &m->map[pos];
    const int32_t off = s->ctx % m->block_size;
    int32_t src = -1, dst = -1;
    if (off == 0) {
        /* last block full (or no block yet): a fresh block extends the table */
        if (!ensure_table_cap(s, s->n_blocks + 1)) return PKV_ERR_BAD_STATE;
        int32_t b = alloc_one(m);
        if (b < 0) {
            m->alloc_failures++;
            m->append_oom++;
            return PKV_ERR_NO_BLOCKS;
        }
        s->table[s->n_blocks++] = b;
        *slot = (int64_t)b * m->block_size;
    } else {
        int32_t tail = s->table[s->n_blocks - 1];
        if (m->ref[tail] == 1) {
            *slot = (int64_t)tail * m->block_size + off;
        } else {
            /* shared, partially filled last block: copy on write */
            int32_t b = alloc_one(m);
            if (b < 0) {
                m->alloc_failures++;
                m->append_oom++;
                return PKV_ERR_NO_BLOCKS;
            }
            m->ref[tail]--;
            s->table[s->n_blocks - 1] = b;
            m->cow_copies++;
            src = tail;
            dst = b;
            *slot = (int64_t)b * m->block_size + off;
        }
    }
    s->ctx++;
    if (cow_src) *cow_src = src;
    if (cow_dst) *cow_dst = dst;
    return PKV_OK;
}

int pkv_mgr_extend(pkv_mgr* m, int64_t seq_id, int32_t n_tokens, int64_t* slots_out, int32_t* cow_src,
                   int32_t* cow_dst) {
    if (!m || n_tokens < 0 || (n_tokens > 0 && !slots_out)) return PKV_ERR_INVALID_ARG;
    int64_t pos = map_find(m, seq_id);
    if (pos < 0) return PKV_ERR_INVALID_ARG;
    if (cow_src) *cow_src = -1;
    if (cow_dst) *cow_dst = -1;
    if (n_tokens == 0) return PKV_OK;
    seq_rec* s = &m->map[pos];
    const int32_t off = s->ctx % m->block_size;
    const int cow = off != 0 && m->ref[s->table[s->n_blocks - 1]] > 1;
    const int64_t end = (int64_t)s->ctx + n_tokens;
    if (end > INT32_MAX) return PKV_ERR_INVALID_ARG;
    const int32_t total = blocks_for(m, end);
    const int32_t fresh = total - s->n_blocks;
    if ((int64_t)fresh + cow > m->n_free) {
        m->alloc_failures++;
        m->append_oom++;
        return PKV_ERR_NO_BLOCKS;
    }
    if (!ensure_table_cap(s, total)) return PKV_ERR_BAD_STATE;
    /* allocation order of n successive appends: the copy of a shared tail first, then fresh blocks */
    int32_t cow_block = -1;
    if (cow) {
        cow_block = alloc_one(m);
        if (cow_block < 0) {
            m->alloc_failures++;
            m->append_oom++;
            return PKV_ERR_NO_BLOCKS;
        }
    }
    for (int32_t i = 0; i < fresh; ++i) {
        int32_t b = alloc_one(m);
        if (b < 0) { /* injected failure: undo in reverse so the free list is restored exactly */
            for (int32_t k = i - 1; k >= 0; --k) {
                m->ref[s->table[s->n_blocks + k]] = 0;
                ring_push_front(m, s->table[s->n_blocks + k]);
            }
            if (cow_block >= 0) {
                m->ref[cow_block] = 0;
                ring_push_front(m, cow_block);
            }
            m->alloc_failures++;
            m->append_oom++;
            return PKV_ERR_NO_BLOCKS;
        }
        s->table[s->n_blocks + i] = b;
    }
    if (cow_block >= 0) {
        const int32_t tail = s->table[s->n_blocks - 1];
        m->ref[tail]--;
        s->table[s->n_blocks - 1] = cow_block;
        m->cow_copies++;
        if (cow_src) *cow_src = tail;
        if (cow_dst) *cow_dst = cow_block;
    }
    s->n_blocks = total;
    for (int32_t i = 0; i < n_tokens; ++i) {
        const int64_t p = (int64_t)s->ctx + i;
        slots_out[i] = (int64_t)s->table[p / m->block_size] * m->block_size + p % m->block_size;
    }
    s->ctx = (int32_t)end;
    return PKV_OK;
}

int pkv_mgr_append_batch(pkv_mgr* m, const int64_t* seq_ids, int32_t n, int64_t* slots_out,
                         int32_t* cow_pairs_out, int32_t* n_cow, int32_t* n_done) {
    if (!m || n < 0 || (n > 0 && (!seq_ids || !slots_out || !cow_pairs_out))) return PKV_ERR_INVALID_ARG;
    int32_t nc = 0, i = 0;
    int rc = PKV_OK;
    for (; i < n; ++i) {
        int32_t src, dst;
        rc = pkv_mgr_append_slot(m, seq_ids[i], &slots_out[i], &src, &dst);
        if (rc != PKV_OK) break;
        if (src >= 0) {
            cow_pairs_out[2 * nc] = src;
            cow_pairs_out[2 * nc + 1] = dst;
            nc++;
        }
    }
    if (n_cow) *n_cow = nc;
    if (n_done) *n_done = i;
    return rc;
}

int pkv_mgr_free_seq(pkv_mgr* m, int64_t seq_id) {
    if (!m) return PKV_ERR_INVALID_ARG;
    int64_t pos = map_find(m, seq_id);
    if (pos < 0) return PKV_ERR_INVALID_ARG;
    seq_rec* s = &m->map[pos];
    for (int32_t i = 0; i < s->n_blocks; ++i) {
        int32_t b = s->table[i];
        if (m->ref[b] <= 0) return PKV_ERR_BAD_STATE; /* cannot happen: refcounts are conserved */
    }
    for (int32_t i = 0; i < s->n_blocks; ++i) {
        int32_t b = s->table[i];
        if (--m->ref[b] == 0) ring_push_back(m, b);
    }
    free(s->table);
    map_erase(m, pos);
    return PKV_OK;
}

int pkv_mgr_block_table(const pkv_mgr* m, int64_t seq_id, int32_t* out, int32_t cap, int32_t* n_blocks,
                        int32_t* ctx_len) {
    if (!m) return PKV_ERR_INVALID_ARG;
    int64_t pos = map_find(m, seq_id);
    if (pos < 0) return PKV_ERR_INVALID_ARG;
    const seq_rec* s = &m->map[pos];
    if (n_blocks) *n_blocks = s->n_blocks;
    if (ctx_len) *ctx_len = s->ctx;
    if (s->n_blocks > cap || (s->n_blocks > 0 && !out)) return PKV_ERR_INVALID_ARG;
    if (s->n_blocks) memcpy(out, s->table, sizeof(int32_t) * (size_t)s->n_blocks);
    return PKV_OK;
}

int pkv_mgr_pack_tables(const pkv_mgr* m, const int64_t* seq_ids, int32_t n, int32_t max_blocks,
                        int32_t* tables_out, int32_t* lens_out) {
    if (!m || n < 0 || max_blocks <= 0 || (n > 0 && (!seq_ids || !tables_out || !lens_out)))
        return PKV_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) {
        int64_t pos = map_find(m, seq_ids[i]);
        if (pos < 0 || m->map[pos].n_blocks > max_blocks) return PKV_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < n; ++i) {
        const seq_rec* s = &m->map[map_find(m, seq_ids[i])];
        int32_t* row = tables_out + (size_t)i * max_blocks;
        if (s->n_blocks) memcpy(row, s->table, sizeof(int32_t) * (size_t)s->n_blocks);
        for (int32_t j = s->n_blocks; j < max_blocks; ++j) row[j] = -1;
        lens_out[i] = s->ctx;
    }
    return PKV_OK;
}

int pkv_mgr_stats(const pkv_mgr* m, pkv_stats* out) {
    if (!m || !out) return PKV_ERR_INVALID_ARG;
    int64_t waste = 0;
    for (int64_t i = 0; i < m->map_cap; ++i)
        if (m->map[i].used) waste += (int64_t)m->map[i].n_blocks * m->block_size - m->map[i].ctx;
    out->free_blocks = m->n_free;
    out->used_blocks = m->num_blocks - m->n_free;
    out->n_seqs = m->n_seqs;
    out->alloc_failures = m->alloc_failures;
    out->tail_waste_rows = waste;
    out->prefix_hits = m->prefix_hits;
    out->cow_copies = m->cow_copies;
    out->append_oom = m->append_oom;
    return PKV_OK;
}

int32_t pkv_mgr_refcount(const pkv_mgr* m, int32_t block) {
    if (!m || block < 0 || block >= m->num_blocks) return -1;
    return m->ref[block];
}

int32_t pkv_mgr_free_list(const pkv_mgr* m, int32_t* out, int32_t cap) {
    if (!m) return -1;
    for (int32_t i = 0; i < m->n_free && i < cap; ++i) out[i] = m->ring[(m->head + i) % m->num_blocks];
    return m->n_free;
}

int pkv_mgr_inject_alloc_failure(pkv_mgr* m, int32_t after_n_allocs) {
    if (!m) return PKV_ERR_INVALID_ARG;
    m->inject_after = after_n_allocs < 0 ? -1 : after_n_allocs;
    return PKV_OK;
}

/* ---- checkpoint / resume ------------------------------------------------------------------ */

#define PKV_IMG_MAGIC 0x4d564b50u /* "PKVM" little-endian */
#define PKV_IMG_VERSION 1u

static uint64_t fnv1a64(const uint8_t* p, size_t n) {
    uint64_t h = 0xcbf29ce484222325ull;
    for (size_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= 0x100000001b3ull;
    }
    return h;
}

static void put_u32(uint8_t** w, uint32_t v) {
    for (int i = 0; i < 4; ++i) *(*w)++ = (uint8_t)(v >> (8 * i));
}
static void put_u64(uint8_t** w, uint64_t v) {
    for (int i = 0; i < 8; ++i) *(*w)++ = (uint8_t)(v >> (8 * i));
}
static uint32_t get_u32(const uint8_t** r) {
    uint32_t v = 0;
    for (int i = 0; i < 4; ++i) v |= (uint32_t)(*(*r)++) << (8 * i);
    return v;
}
static uint64_t get_u64(const uint8_t** r) {
    uint64_t v = 0;
    for (int i = 0; i < 8; ++i) v |= (uint64_t)(*(*r)++) << (8 * i);
    return v;
}

size_t pkv_mgr_save_bytes(const pkv_mgr* m) {
    if (!m) return 0;
    size_t n = 4 + 4 + 4 + 4 + 4 + (size_t)m->n_free * 4 + 4 * 8 + 8;
    for (int64_t i = 0; i < m->map_cap; ++i)
        if (m->map[i].used) n += 8 + 4 + 4 + (size_t)m->map[i].n_blocks * 4;
    return n + 8;
}

static int cmp_id(const void* a, const void* b) {
    const int64_t x = (*(const seq_rec* const*)a)->id, y = (*(const seq_rec* const*)b)->id;
    return x < y ? -1 : (x > y);
}

int pkv_mgr_save(const pkv_mgr* m, void* buf, size_t cap, size_t* written) {
    if (!m || !buf || !written) return PKV_ERR_INVALID_ARG;
    const size_t need = pkv_mgr_save_bytes(m);
    if (cap < need) return PKV_ERR_INVALID_ARG;
    const seq_rec** order = NULL;
    if (m->n_seqs > 0) {
        order = (const seq_rec**)malloc(sizeof(seq_rec*) * (size_t)m->n_seqs);
        if (!order) return PKV_ERR_INVALID_ARG;
        int64_t k = 0;
        for (int64_t i = 0; i < m->map_cap; ++i)
            if (m->map[i].used) order[k++] = &m->map[i];
        qsort(order, (size_t)m->n_seqs, sizeof(seq_rec*), cmp_id);
    }
    uint8_t* w = (uint8_t*)buf;
    put_u32(&w, PKV_IMG_MAGIC);
    put_u32(&w, PKV_IMG_VERSION);
    put_u32(&w, (uint32_t)m->num_blocks);
    put_u32(&w, (uint32_t)m->block_size);
    put_u32(&w, (uint32_t)m->n_free);
    for (int32_t i = 0; i < m->n_free; ++i) put_u32(&w, (uint32_t)m->ring[(m->head + i) % m->num_blocks]);
    put_u64(&w, (uint64_t)m->alloc_failures);
    put_u64(&w, (uint64_t)m->prefix_hits);
    put_u64(&w, (uint64_t)m->cow_copies);
    put_u64(&w, (uint64_t)m->append_oom);
    put_u64(&w, (uint64_t)m->n_seqs);
    for (int64_t k = 0; k < m->n_seqs; ++k) {
        const seq_rec* r = order[k];
        put_u64(&w, (uint64_t)r->id);
        put_u32(&w, (uint32_t)r->ctx);
        put_u32(&w, (uint32_t)r->n_blocks);
        for (int32_t b = 0; b < r->n_blocks; ++b) put_u32(&w, (uint32_t)r->table[b]);
    }
    free(order);
    put_u64(&w, fnv1a64((const uint8_t*)buf, (size_t)(w - (uint8_t*)buf)));
    *written = (size_t)(w - (uint8_t*)buf);
    return PKV_OK;
}

pkv_mgr* pkv_mgr_load(const void* buf, size_t len) {
    if (!buf || len < 4 + 4 + 4 + 4 + 4 + 5 * 8 + 8) return NULL;
    const uint8_t* base = (const uint8_t*)buf;
    const uint8_t* end = base + len - 8;
    const uint8_t* sum_at = end;
    if (get_u64(&sum_at) != fnv1a64(base, len - 8)) return NULL;
    const uint8_t* r = base;
    if (get_u32(&r) != PKV_IMG_MAGIC || get_u32(&r) != PKV_IMG_VERSION) return NULL;
    const int32_t num_blocks = (int32_t)get_u32(&r);
    const int32_t block_size = (int32_t)get_u32(&r);
    const int32_t n_free = (int32_t)get_u32(&r);
    if (num_blocks <= 0 || block_size <= 0 || n_free < 0 || n_free > num_blocks) return NULL;
    if ((size_t)(end - r) < (size_t)n_free * 4 + 5 * 8) return NULL;
    pkv_mgr* m = pkv_mgr_create(num_blocks, block_size, NULL);
    if (!m) return NULL;
    /* free list, front first; ref[] temporarily marks "free" with -1 */
    for (int32_t i = 0; i < n_free; ++i) {
        const int32_t b = (int32_t)get_u32(&r);
        if (b < 0 || b >= num_blocks || m->ref[b] != 0) goto bad;
        m->ref[b] = -1;
        m->ring[i] = b;
    }
    m->head = 0;
    m->n_free = n_free;
    m->alloc_failures = (int64_t)get_u64(&r);
    m->prefix_hits = (int64_t)get_u64(&r);
    m->cow_copies = (int64_t)get_u64(&r);
    m->append_oom = (int64_t)get_u64(&r);
    const int64_t n_seqs = (int64_t)get_u64(&r);
    if (n_seqs < 0) goto bad;
    for (int64_t k = 0; k < n_seqs; ++k) {
        if ((size_t)(end - r) < 16) goto bad;
        const int64_t id = (int64_t)get_u64(&r);
        const int32_t ctx = (int32_t)get_u32(&r);
        const int32_t nb = (int32_t)get_u32(&r);
        if (ctx < 0 || nb < 0 || nb != (int32_t)(((int64_t)ctx + block_size - 1) / block_size)) goto bad;
        if ((size_t)(end - r) < (size_t)nb * 4) goto bad;
        if (map_find(m, id) >= 0 || !map_reserve_one(m)) goto bad;
        int32_t* table = NULL;
        if (nb > 0) {
            table = (int32_t*)malloc(sizeof(int32_t) * (size_t)nb);
            if (!table) goto bad;
        }
        for (int32_t b = 0; b < nb; ++b) {
            const int32_t id_b = (int32_t)get_u32(&r);
            if (id_b < 0 || id_b >= num_blocks || m->ref[id_b] < 0) {
                free(table);
                goto bad;
            }
            table[b] = id_b;
            m->ref[id_b]++;
        }
        seq_rec* rec = map_insert(m, id);
        rec->table = table;
        rec->n_blocks = nb;
        rec->cap = nb;
        rec->ctx = ctx;
    }
    if (r != end) goto bad;
    /* every block is either free or held by some table */
    for (int32_t b = 0; b < num_blocks; ++b) {
        if (m->ref[b] == 0) goto bad;
        if (m->ref[b] < 0) m->ref[b] = 0;
    }
    return m;
bad:
    for (int32_t b = 0; b < num_blocks; ++b)
        if (m->ref[b] < 0) m->ref[b] = 0;
    pkv_mgr_destroy(m);
    return NULL;
}
