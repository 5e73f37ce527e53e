// Host half of libpagedattn: block allocator, step metadata, work planning, utilities.
//
// Allocator semantics follow "P3: native paged-KV continuous-batching sampler",
// Design / paged.py (LIFO free list + refcounts, double-free guard, all-or-nothing capacity,
// read-only shared blocks, check_consistent) and Design / engine.py (prefix sharing of full
// blocks). The typed exhaustion error follows "Optional paged KV cache (vLLM-style) - v1
// design", Design.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <unordered_map>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/pagedattn.h"
#include "common.h"

namespace {

thread_local int32_t g_last_cuda_error = 0;

}  // namespace

namespace pa_detail {

int32_t note_cuda(cudaError_t e) {
    if (e == cudaSuccess) return PA_OK;
    g_last_cuda_error = static_cast<int32_t>(e);
    return PA_ERR_CUDA;
}

int32_t check_shape(const pa_shape* s) {
    if (!s) return PA_ERR_INVALID;
    if (s->num_q_heads <= 0 || s->num_kv_heads <= 0 || s->head_dim <= 0 || s->block_size <= 0 ||
        s->num_blocks < 0)
        return PA_ERR_INVALID;
    if (s->num_q_heads % s->num_kv_heads) return PA_ERR_SHAPE;
    const int g = s->num_q_heads / s->num_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return PA_ERR_SHAPE;
    if (s->head_dim != 64 && s->head_dim != 128) return PA_ERR_SHAPE;
    const int bs = s->block_size;
    if (bs < 8 || bs > 128 || (bs & (bs - 1))) return PA_ERR_SHAPE;
    return PA_OK;
}

int32_t check_step_meta(int32_t B, const int32_t* cu, const int32_t* ctx) {
    if (B < 0) return PA_ERR_INVALID;
    if (B > 0 && (!cu || !ctx)) return PA_ERR_INVALID;
    if (B == 0) return (cu && cu[0] != 0) ? PA_ERR_INVALID : PA_OK;
    if (cu[0] != 0) return PA_ERR_INVALID;
    for (int32_t s = 0; s < B; ++s) {
        const int64_t n = int64_t(cu[s + 1]) - cu[s];
        if (n < 0) return PA_ERR_INVALID;
        if (ctx[s] < 0 || n > ctx[s]) return PA_ERR_INVALID;
    }
    return PA_OK;
}

}  // namespace pa_detail

using namespace pa_detail;

// ------------------------------------------------------------------------- allocator

struct pa_allocator {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    std::vector<int32_t> free_stack;      // top = back()
    std::vector<int32_t> ref;
    std::unordered_map<int32_t, std::vector<int32_t>> tables;
};

extern "C" {

int32_t pa_abi_version(void) { return 3; }

const char* pa_status_string(int32_t st) {
    switch (st) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID: return "PA_ERR_INVALID";
        case PA_ERR_SHAPE: return "PA_ERR_SHAPE";
        case PA_ERR_BOUNDS: return "PA_ERR_BOUNDS";
        case PA_ERR_OOM: return "PA_ERR_OOM";
        case PA_ERR_READONLY: return "PA_ERR_READONLY";
        case PA_ERR_DOUBLE_FREE: return "PA_ERR_DOUBLE_FREE";
        case PA_ERR_INCONSISTENT: return "PA_ERR_INCONSISTENT";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_STATE: return "PA_ERR_STATE";
        default: return "PA_ERR_UNKNOWN";
    }
}

int32_t pa_last_cuda_error(void) { return g_last_cuda_error; }

int32_t pa_device_sm_count(int32_t* n) {
    if (!n) return PA_ERR_INVALID;
    int dev = 0;
    int32_t st = note_cuda(cudaGetDevice(&dev));
    if (st) return st;
    int v = 0;
    st = note_cuda(cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev));
    if (st) return st;
    *n = v;
    return PA_OK;
}

int32_t pa_alloc_create(int32_t num_blocks, int32_t block_size, pa_allocator** out) {
    if (!out || num_blocks < 0 || block_size <= 0) return PA_ERR_INVALID;
    auto* a = new pa_allocator;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->ref.assign(num_blocks, 0);
    a->free_stack.resize(num_blocks);
    for (int32_t i = 0; i < num_blocks; ++i) a->free_stack[i] = num_blocks - 1 - i;
    *out = a;
    return PA_OK;
}

int32_t pa_alloc_destroy(pa_allocator* a) {
    delete a;
    return PA_OK;
}

int32_t pa_alloc_block(pa_allocator* a, int32_t* block) {
    if (!a || !block) return PA_ERR_INVALID;
    if (a->free_stack.empty()) return PA_ERR_OOM;
    const int32_t b = a->free_stack.back();
    a->free_stack.pop_back();
    a->ref[b] = 1;
    *block = b;
    return PA_OK;
}

int32_t pa_alloc_incref(pa_allocator* a, int32_t b) {
    if (!a) return PA_ERR_INVALID;
    if (b < 0 || b >= a->num_blocks) return PA_ERR_BOUNDS;
    if (a->ref[b] <= 0) return PA_ERR_STATE;
    a->ref[b] += 1;
    return PA_OK;
}

int32_t pa_alloc_free_block(pa_allocator* a, int32_t b) {
    if (!a) return PA_ERR_INVALID;
    if (b < 0 || b >= a->num_blocks) return PA_ERR_BOUNDS;
    if (a->ref[b] == 0) return PA_ERR_DOUBLE_FREE;
    if (--a->ref[b] == 0) a->free_stack.push_back(b);
    return PA_OK;
}

static int64_t blocks_for(int64_t n_tokens, int32_t bs) { return (n_tokens + bs - 1) / bs; }

int32_t pa_alloc_admit(pa_allocator* a, int32_t seq, int32_t n_tokens, int32_t share_src,
                       int32_t n_shared) {
    if (!a || seq < 0 || n_tokens < 0 || n_shared < 0) return PA_ERR_INVALID;
    if (a->tables.count(seq)) return PA_ERR_STATE;
    const std::vector<int32_t>* src = nullptr;
    if (share_src >= 0 && n_shared > 0) {
        auto it = a->tables.find(share_src);
        if (it == a->tables.end()) return PA_ERR_STATE;
        src = &it->second;
        if (n_shared > int32_t(src->size()) || int64_t(n_shared) * a->block_size > n_tokens)
            return PA_ERR_INVALID;
    } else {
        n_shared = 0;
    }
    const int64_t need = blocks_for(n_tokens, a->block_size) - n_shared;
    if (need > int64_t(a->free_stack.size())) return PA_ERR_OOM;
    std::vector<int32_t> t;
    t.reserve(n_shared + std::max<int64_t>(need, 0));
    for (int32_t i = 0; i < n_shared; ++i) {
        const int32_t b = (*src)[i];
        a->ref[b] += 1;
        t.push_back(b);
    }
    for (int64_t i = 0; i < need; ++i) {
        int32_t b;
        pa_alloc_block(a, &b);
        t.push_back(b);
    }
    a->tables.emplace(seq, std::move(t));
    return PA_OK;
}

int32_t pa_alloc_ensure_capacity(pa_allocator* a, int32_t seq, int32_t n_tokens) {
    if (!a || n_tokens < 0) return PA_ERR_INVALID;
    auto it = a->tables.find(seq);
    if (it == a->tables.end()) return PA_ERR_STATE;
    const int64_t need = blocks_for(n_tokens, a->block_size) - int64_t(it->second.size());
    if (need <= 0) return PA_OK;
    if (need > int64_t(a->free_stack.size())) return PA_ERR_OOM;
    for (int64_t i = 0; i < need; ++i) {
        int32_t b;
        pa_alloc_block(a, &b);
        it->second.push_back(b);
    }
    return PA_OK;
}

int32_t pa_alloc_free_seq(pa_allocator* a, int32_t seq) {
    if (!a) return PA_ERR_INVALID;
    auto it = a->tables.find(seq);
    if (it == a->tables.end()) return PA_ERR_STATE;
    for (int32_t b : it->second) {
        const int32_t st = pa_alloc_free_block(a, b);
        if (st) return st;
    }
    a->tables.erase(it);
    return PA_OK;
}

int32_t pa_alloc_trim(pa_allocator* a, int32_t seq, int32_t n_tokens) {
    if (!a || n_tokens < 0) return PA_ERR_INVALID;
    auto it = a->tables.find(seq);
    if (it == a->tables.end()) return PA_ERR_STATE;
    std::vector<int32_t>& t = it->second;
    const int64_t keep = blocks_for(n_tokens, a->block_size);
    if (keep > int64_t(t.size())) return PA_ERR_BOUNDS;
    // the tail goes back last block first, so the block next to the kept part is reused first
    while (int64_t(t.size()) > keep) {
        const int32_t st = pa_alloc_free_block(a, t.back());
        if (st) return st;
        t.pop_back();
    }
    return PA_OK;
}

int32_t pa_alloc_fork(pa_allocator* a, int32_t src, int32_t dst) {
    if (!a || dst < 0) return PA_ERR_INVALID;
    if (a->tables.count(dst)) return PA_ERR_STATE;
    auto it = a->tables.find(src);
    if (it == a->tables.end()) return PA_ERR_STATE;
    for (int32_t b : it->second) a->ref[b] += 1;
    std::vector<int32_t> copy = it->second;
    a->tables.emplace(dst, std::move(copy));
    return PA_OK;
}

int32_t pa_alloc_cow(pa_allocator* a, int32_t seq, int32_t start, int32_t n, int32_t* pairs,
                     int32_t max_pairs, int32_t* n_pairs) {
    if (!a || !n_pairs || n < 0 || start < 0 || max_pairs < 0) return PA_ERR_INVALID;
    auto it = a->tables.find(seq);
    if (it == a->tables.end()) return PA_ERR_STATE;
    std::vector<int32_t>& t = it->second;
    *n_pairs = 0;
    if (n == 0) return PA_OK;
    const int64_t first = int64_t(start) / a->block_size;
    const int64_t last = (int64_t(start) + n - 1) / a->block_size;
    if (last >= int64_t(t.size())) return PA_ERR_BOUNDS;
    int32_t shared = 0;
    for (int64_t j = first; j <= last; ++j) shared += a->ref[t[j]] > 1;
    if (shared > max_pairs || (shared > 0 && !pairs)) return PA_ERR_INVALID;
    if (shared > int32_t(a->free_stack.size())) return PA_ERR_OOM;
    int32_t k = 0;
    for (int64_t j = first; j <= last; ++j) {
        if (a->ref[t[j]] <= 1) continue;
        int32_t fresh;
        pa_alloc_block(a, &fresh);
        const int32_t old = t[j];
        a->ref[old] -= 1;                 // this table's reference only: still > 0
        t[j] = fresh;
        pairs[2 * k] = old;
        pairs[2 * k + 1] = fresh;
        ++k;
    }
    *n_pairs = k;
    return PA_OK;
}

int32_t pa_alloc_check_consistent(const pa_allocator* a) {
    if (!a) return PA_ERR_INVALID;
    std::vector<uint8_t> on_free(a->num_blocks, 0);
    for (int32_t b : a->free_stack) {
        if (b < 0 || b >= a->num_blocks || on_free[b]) return PA_ERR_INCONSISTENT;
        on_free[b] = 1;
        if (a->ref[b] != 0) return PA_ERR_INCONSISTENT;
    }
    int64_t referenced = 0;
    for (int32_t b = 0; b < a->num_blocks; ++b) referenced += a->ref[b] > 0;
    if (referenced + int64_t(a->free_stack.size()) != a->num_blocks) return PA_ERR_INCONSISTENT;
    std::vector<int32_t> want(a->num_blocks, 0);
    for (const auto& kv : a->tables)
        for (int32_t b : kv.second) {
            if (b < 0 || b >= a->num_blocks) return PA_ERR_INCONSISTENT;
            want[b] += 1;
        }
    for (int32_t b = 0; b < a->num_blocks; ++b)
        if (want[b] != a->ref[b]) return PA_ERR_INCONSISTENT;
    return PA_OK;
}

int32_t pa_alloc_num_free(const pa_allocator* a) {
    return a ? int32_t(a->free_stack.size()) : -1;
}

int32_t pa_alloc_refcount(const pa_allocator* a, int32_t b) {
    if (!a || b < 0 || b >= a->num_blocks) return -1;
    return a->ref[b];
}

int32_t pa_alloc_table(const pa_allocator* a, int32_t seq, int32_t* out, int32_t cap,
                       int32_t* n) {
    if (!a || !n || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID;
    auto it = a->tables.find(seq);
    if (it == a->tables.end()) return PA_ERR_STATE;
    const int32_t len = int32_t(it->second.size());
    *n = len;
    std::memcpy(out, it->second.data(), sizeof(int32_t) * std::min(cap, len));
    return PA_OK;
}

static int32_t slots_of(const pa_allocator* a, const std::vector<int32_t>& t, int32_t start,
                        int32_t n, int32_t* out) {
    const int32_t bs = a->block_size;
    for (int32_t i = 0; i < n; ++i) {
        const int64_t p = int64_t(start) + i;
        const int64_t j = p / bs;
        if (p < 0 || j >= int64_t(t.size())) return PA_ERR_BOUNDS;
        if (a->ref[t[j]] > 1) return PA_ERR_READONLY;
    }
    for (int32_t i = 0; i < n; ++i) {
        const int64_t p = int64_t(start) + i;
        out[i] = int32_t(int64_t(t[p / bs]) * bs + p % bs);
    }
    return PA_OK;
}

int32_t pa_alloc_slots(const pa_allocator* a, int32_t seq, int32_t start, int32_t n,
                       int32_t* out) {
    if (!a || n < 0 || (n > 0 && !out)) return PA_ERR_INVALID;
    auto it = a->tables.find(seq);
    if (it == a->tables.end()) return PA_ERR_STATE;
    return slots_of(a, it->second, start, n, out);
}

int32_t pa_alloc_build_step(const pa_allocator* a, const int32_t* seqs, const int32_t* ctx_lens,
                            const int32_t* n_new, int32_t B, int32_t* cu_seqlens_q,
                            int32_t* slot_mapping, int32_t* block_table, int32_t max_blocks) {
    if (!a || B < 0 || max_blocks <= 0 || !cu_seqlens_q) return PA_ERR_INVALID;
    if (B > 0 && (!seqs || !ctx_lens || !n_new || !block_table)) return PA_ERR_INVALID;
    // validate everything before writing anything
    int64_t T = 0;
    std::vector<const std::vector<int32_t>*> rows(B);
    for (int32_t i = 0; i < B; ++i) {
        auto it = a->tables.find(seqs[i]);
        if (it == a->tables.end()) return PA_ERR_STATE;
        if (ctx_lens[i] < 0 || n_new[i] < 0 || n_new[i] > ctx_lens[i]) return PA_ERR_INVALID;
        const int64_t nb = blocks_for(ctx_lens[i], a->block_size);
        if (nb > int64_t(it->second.size())) return PA_ERR_BOUNDS;
        if (nb > max_blocks) return PA_ERR_BOUNDS;
        const int32_t start = ctx_lens[i] - n_new[i];
        for (int32_t k = 0; k < n_new[i]; ++k) {
            const int64_t j = (int64_t(start) + k) / a->block_size;
            if (a->ref[it->second[j]] > 1) return PA_ERR_READONLY;
        }
        rows[i] = &it->second;
        T += n_new[i];
    }
    if (T > INT32_MAX) return PA_ERR_INVALID;
    if (T > 0 && !slot_mapping) return PA_ERR_INVALID;
    cu_seqlens_q[0] = 0;
    for (int32_t i = 0; i < B; ++i) {
        cu_seqlens_q[i + 1] = cu_seqlens_q[i] + n_new[i];
        int32_t* row = block_table + int64_t(i) * max_blocks;
        const int64_t nb = blocks_for(ctx_lens[i], a->block_size);
        for (int32_t j = 0; j < max_blocks; ++j) row[j] = j < nb ? (*rows[i])[j] : -1;
        slots_of(a, *rows[i], ctx_lens[i] - n_new[i], n_new[i], slot_mapping + cu_seqlens_q[i]);
    }
    return PA_OK;
}

// --------------------------------------------------------------------- step metadata

int32_t pa_compute_slots(const pa_shape* shape, const int32_t* block_table, int32_t B,
                         int32_t max_blocks, const int32_t* cu, const int32_t* ctx,
                         int32_t* slot_mapping) {
    int32_t st = check_shape(shape);
    if (st) return st;
    st = check_step_meta(B, cu, ctx);
    if (st) return st;
    if (B > 0 && (!block_table || max_blocks <= 0)) return PA_ERR_INVALID;
    const int32_t bs = shape->block_size;
    for (int32_t s = 0; s < B; ++s) {
        const int64_t nb = blocks_for(ctx[s], bs);
        if (nb > max_blocks) return PA_ERR_BOUNDS;
        for (int64_t j = 0; j < nb; ++j) {
            const int32_t b = block_table[int64_t(s) * max_blocks + j];
            if (b < 0 || b >= shape->num_blocks) return PA_ERR_BOUNDS;
        }
    }
    const int32_t T = B > 0 ? cu[B] : 0;
    if (T > 0 && !slot_mapping) return PA_ERR_INVALID;
    for (int32_t s = 0; s < B; ++s) {
        const int32_t n = cu[s + 1] - cu[s];
        for (int32_t i = 0; i < n; ++i) {
            const int64_t p = int64_t(ctx[s]) - n + i;
            const int64_t b = block_table[int64_t(s) * max_blocks + p / bs];
            slot_mapping[cu[s] + i] = int32_t(b * bs + p % bs);
        }
    }
    return PA_OK;
}

int64_t pa_plan_max_items(const pa_shape* shape, int32_t B, int32_t T, int32_t max_ctx) {
    if (check_shape(shape) || B < 0 || T < 0 || max_ctx < 0) return 0;
    const int32_t g = shape->num_q_heads / shape->num_kv_heads;
    const int64_t rows_per_tile = PA_ROWS / g;
    const int64_t tiles = int64_t(B) + T / rows_per_tile + 1;   // each seq adds <= 1 ragged tile
    const int64_t splits = (int64_t(max_ctx) + PA_SPLIT_TOKENS - 1) / PA_SPLIT_TOKENS;
    return tiles * shape->num_kv_heads * std::max<int64_t>(splits, 1);
}

namespace {

// A unit of the deal: items [first, first + count) of the generated items, which go to one
// list, consecutively, in this order (one item, or a group's GROUP item and its RESUMEs).
struct Unit {
    int32_t first, count;
    int64_t cost;       // sum over its items of n_tiles + 1
};

// The PLAIN items of query-row tile [t0, t0 + nt) of sequence s, KV heads all, splits from
// sp_first on: a decode row's splits go to separate items; a prefill tile keeps all of its
// splits in one item and folds them in the kernel.
void plain_items(const pa_shape* shape, int32_t s, int32_t q0, int32_t n, int32_t t0, int32_t nt,
                 const int32_t* ctx, int32_t sp_first, std::vector<pa_work_item>& out,
                 std::vector<Unit>& units) {
    const int64_t p_max = int64_t(ctx[s]) - n + t0 + nt - 1;
    const int32_t nsplit = int32_t(p_max / PA_SPLIT_TOKENS + 1);
    const int32_t per_item = n > 1 ? nsplit : 1;
    for (int32_t h = 0; h < shape->num_kv_heads; ++h)
        for (int32_t sp = sp_first; sp < nsplit; sp += per_item) {
            const int64_t k0 = int64_t(sp) * PA_SPLIT_TOKENS;
            const int64_t k1 = std::min<int64_t>(k0 + int64_t(per_item) * PA_SPLIT_TOKENS, p_max + 1);
            pa_work_item it{};
            it.seq = s;
            it.q_start = q0 + t0;
            it.n_q = nt;
            it.kv_head = h;
            it.split = sp;
            it.n_tiles = int32_t((k1 - k0 + PA_TILE_KEYS - 1) / PA_TILE_KEYS);
            it.n_splits = per_item;
            it.kind = PA_ITEM_PLAIN;
            units.push_back({int32_t(out.size()), 1, int64_t(it.n_tiles) + 1});
            out.push_back(it);
        }
}

// Deals the units longest processing time first: each unit, by decreasing cost (ties in
// generation order), joins the list (one per CTA) with the least cost so far, the lower list on
// a tie; its items take consecutive places in that list. The output holds the first item of
// every list (list c at index c), then the second item of every list that has one, in list
// order, and so on, with `next` linking each list. The kernel runs min(output items,
// PA_PLAN_CTAS) CTAs, CTA c from index c: when units make fewer lists G than that, padding
// items (n_q == 0) take indices G .. PA_PLAN_CTAS - 1, so that the CTAs past the lists find
// no work.
int32_t deal(const std::vector<pa_work_item>& out, const std::vector<Unit>& units,
             pa_work_item* items, int32_t max_items, int32_t* n_items) {
    const int32_t n = int32_t(out.size());
    const int32_t nu = int32_t(units.size());
    const int32_t G = std::min<int32_t>(nu, PA_PLAN_CTAS);
    const int32_t pad = G < std::min<int32_t>(n, PA_PLAN_CTAS) ? PA_PLAN_CTAS - G : 0;
    if (int64_t(n) + pad > max_items) return PA_ERR_INVALID;
    // by decreasing cost, ties in generation order (a stable counting sort when it is small)
    int64_t max_cost = 0;
    for (const Unit& u : units) max_cost = std::max(max_cost, u.cost);
    std::vector<int32_t> by_cost(static_cast<size_t>(nu));
    if (max_cost <= 4 * int64_t(nu) + 4096) {
        std::vector<int32_t> first(size_t(max_cost) + 2, 0);
        for (const Unit& u : units) ++first[size_t(max_cost - u.cost) + 1];
        for (size_t k = 1; k < first.size(); ++k) first[k] += first[k - 1];
        for (int32_t i = 0; i < nu; ++i)
            by_cost[size_t(first[size_t(max_cost - units[size_t(i)].cost)]++)] = i;
    } else {
        for (int32_t i = 0; i < nu; ++i) by_cost[size_t(i)] = i;
        std::stable_sort(by_cost.begin(), by_cost.end(), [&](int32_t x, int32_t y) {
            return units[size_t(x)].cost > units[size_t(y)].cost;
        });
    }
    // a binary min-heap of keys cost * 256 + list (G <= 256), so that equal costs order by list
    static_assert(PA_PLAN_CTAS <= 256, "list index must fit the heap key's low byte");
    std::vector<uint64_t> heap(static_cast<size_t>(G));
    for (int32_t c = 0; c < G; ++c) heap[size_t(c)] = uint64_t(c);   // ascending: a heap
    std::vector<int32_t> owner(static_cast<size_t>(n)), rank(static_cast<size_t>(n));
    std::vector<int32_t> len(static_cast<size_t>(G), 0);
    for (int32_t j = 0; j < nu && G > 0; ++j) {
        const Unit& u = units[size_t(by_cost[size_t(j)])];
        const int32_t c = int32_t(heap[0] & 255u);
        for (int32_t k = 0; k < u.count; ++k) {
            owner[size_t(u.first + k)] = c;
            rank[size_t(u.first + k)] = len[size_t(c)]++;
        }
        uint64_t key = heap[0] + uint64_t(u.cost) * 256u;
        size_t k = 0;                                                // sift the root down
        for (;;) {
            size_t m = 2 * k + 1;
            if (m >= heap.size()) break;
            if (m + 1 < heap.size() && heap[m + 1] < heap[m]) ++m;
            if (heap[m] >= key) break;
            heap[k] = heap[m];
            k = m;
        }
        heap[k] = key;
    }
    // stored position by position: so list c starts at index c and a successor has a higher
    // index
    std::vector<int32_t> off(size_t(G) + 1, 0);
    int32_t longest = 0;
    for (int32_t c = 0; c < G; ++c) {
        off[size_t(c) + 1] = off[size_t(c)] + len[size_t(c)];
        longest = std::max(longest, len[size_t(c)]);
    }
    std::vector<int32_t> member(static_cast<size_t>(n)), at(static_cast<size_t>(n));
    for (int32_t i = 0; i < n; ++i)
        member[size_t(off[size_t(owner[size_t(i)])] + rank[size_t(i)])] = i;
    int32_t pos = 0;
    for (int32_t k = 0; k < longest; ++k) {
        for (int32_t c = 0; c < G; ++c)
            if (k < len[size_t(c)]) at[size_t(member[size_t(off[size_t(c)] + k)])] = pos++;
        if (k == 0) {
            for (int32_t j = 0; j < pad; ++j) items[pos + j] = pa_work_item{};   // n_q == 0
            pos += pad;
        }
    }
    for (int32_t i = 0; i < n; ++i) {
        const int32_t c = owner[size_t(i)], k = rank[size_t(i)];
        pa_work_item it = out[size_t(i)];
        it.next = k + 1 < len[size_t(c)] ? at[size_t(member[size_t(off[size_t(c)] + k + 1)])] : -1;
        items[at[size_t(i)]] = it;
    }
    *n_items = n + pad;
    return PA_OK;
}

int32_t plan(const pa_shape* shape, int32_t B, const int32_t* cu, const int32_t* ctx,
             const int32_t* table, int32_t max_blocks, pa_work_item* items, int32_t max_items,
             int32_t* n_items) {
    int32_t st = check_shape(shape);
    if (st) return st;
    st = check_step_meta(B, cu, ctx);
    if (st) return st;
    if (!n_items || max_items < 0 || (max_items > 0 && !items)) return PA_ERR_INVALID;
    const int32_t g = shape->num_q_heads / shape->num_kv_heads;
    const int32_t rpt = PA_ROWS / g;
    const int32_t bs = shape->block_size;
    if (table) {
        if (max_blocks < 0) return PA_ERR_INVALID;
        for (int32_t s = 0; s < B; ++s)
            if ((int64_t(ctx[s]) + bs - 1) / bs > max_blocks) return PA_ERR_BOUNDS;
    }
    std::vector<pa_work_item> out;
    std::vector<Unit> units;
    out.reserve(size_t(std::min<int64_t>(max_items, 1 << 16)));
    const auto decode = [&](int32_t s) { return cu[s + 1] - cu[s] == 1; };
    // the leading key tiles of split 0 that a row at ctx has keys past (the rest of its split
    // 0 is left for a RESUME item)
    const auto tile_cap = [&](int32_t s) {
        return std::min<int32_t>(PA_SPLIT_TOKENS / PA_TILE_KEYS - 1, (ctx[s] - 1) / PA_TILE_KEYS);
    };
    const int32_t blocks_per_tile = PA_TILE_KEYS / bs;
    const auto common = [&](int32_t a, int32_t b, int32_t bound) {
        const int32_t* ra = table + int64_t(a) * max_blocks;
        const int32_t* rb = table + int64_t(b) * max_blocks;
        int32_t t = 0;
        while (t < bound &&
               std::memcmp(ra + int64_t(t) * blocks_per_tile, rb + int64_t(t) * blocks_per_tile,
                           size_t(blocks_per_tile) * 4) == 0)
            ++t;
        return t;
    };
    for (int32_t s = 0; s < B;) {
        // a run of decode rows that share at least two leading tiles with its first row
        int32_t e = s + 1, shared = 0;
        if (table && decode(s)) {
            shared = tile_cap(s);
            while (e < B && decode(e) && (e - s + 1) * g <= PA_ROWS) {
                const int32_t c = common(s, e, std::min(shared, tile_cap(e)));
                if (c < 2) break;
                shared = c;
                ++e;
            }
        }
        if (e - s < 2 || shared < 2) {
            const int32_t n = cu[s + 1] - cu[s];
            for (int32_t t0 = 0; t0 < n; t0 += rpt)
                plain_items(shape, s, cu[s], n, t0, std::min(rpt, n - t0), ctx, 0, out, units);
            ++s;
            continue;
        }
        for (int32_t h = 0; h < shape->num_kv_heads; ++h) {
            Unit u{int32_t(out.size()), 0, 0};
            pa_work_item it{};
            it.seq = s;
            it.q_start = cu[s];
            it.n_q = e - s;
            it.kv_head = h;
            it.split = 0;
            it.n_tiles = shared;
            it.n_splits = 1;
            it.kind = PA_ITEM_GROUP;
            it.tile0 = shared;
            out.push_back(it);
            u.cost += int64_t(it.n_tiles) + 1;
            for (int32_t m = s; m < e; ++m) {
                pa_work_item r{};
                r.seq = m;
                r.q_start = cu[m];
                r.n_q = 1;
                r.kv_head = h;
                r.split = 0;
                r.n_tiles = (std::min(ctx[m], PA_SPLIT_TOKENS) + PA_TILE_KEYS - 1) / PA_TILE_KEYS -
                            shared;
                r.n_splits = 1;
                r.kind = PA_ITEM_RESUME;
                r.tile0 = shared;
                out.push_back(r);
                u.cost += int64_t(r.n_tiles) + 1;
            }
            u.count = int32_t(out.size()) - u.first;
            units.push_back(u);
        }
        for (int32_t m = s; m < e; ++m) plain_items(shape, m, cu[m], 1, 0, 1, ctx, 1, out, units);
        s = e;
    }
    if (int64_t(out.size()) > max_items) return PA_ERR_INVALID;
    return deal(out, units, items, max_items, n_items);
}

}  // namespace

int32_t pa_plan_step(const pa_shape* shape, int32_t B, const int32_t* cu, const int32_t* ctx,
                     pa_work_item* items, int32_t max_items, int32_t* n_items) {
    return plan(shape, B, cu, ctx, nullptr, 0, items, max_items, n_items);
}

int64_t pa_plan_max_items_shared(const pa_shape* shape, int32_t B, int32_t T, int32_t max_ctx) {
    const int64_t n = pa_plan_max_items(shape, B, T, max_ctx);
    if (n <= 0) return n;
    // at most one GROUP item per KV head for every two sequences, and the padding that keeps
    // the CTAs past a plan's lists idle
    return n + int64_t(B / 2) * shape->num_kv_heads + PA_PLAN_CTAS;
}

int32_t pa_plan_step_shared(const pa_shape* shape, int32_t B, const int32_t* cu,
                            const int32_t* ctx, const int32_t* block_table, int32_t max_blocks,
                            pa_work_item* items, int32_t max_items, int32_t* n_items) {
    if (!block_table && B > 0) return PA_ERR_INVALID;
    return plan(shape, B, cu, ctx, block_table, max_blocks, items, max_items, n_items);
}

size_t pa_workspace_bytes(const pa_shape* shape, int32_t T, int32_t max_ctx) {
    if (check_shape(shape) || T < 0 || max_ctx < 0) return 0;
    const size_t splits = (size_t(max_ctx) + PA_SPLIT_TOKENS - 1) / PA_SPLIT_TOKENS;
    const size_t per = size_t(shape->num_q_heads) * (shape->head_dim + 2) * sizeof(float);
    return std::max<size_t>(size_t(T) * std::max<size_t>(splits, 1) * per, 256);
}

int32_t pa_upload_block_table(const pa_shape* shape, const int32_t* host, int32_t* dev,
                              int32_t B, int32_t max_blocks, pa_stream_t stream) {
    int32_t st = check_shape(shape);
    if (st) return st;
    if (B < 0 || max_blocks < 0) return PA_ERR_INVALID;
    const int64_t n = int64_t(B) * max_blocks;
    if (n == 0) return PA_OK;
    if (!host) return PA_ERR_INVALID;
    for (int64_t i = 0; i < n; ++i)
        if (host[i] < -1 || host[i] >= shape->num_blocks) return PA_ERR_BOUNDS;
    if (!dev) return PA_ERR_INVALID;
    return note_cuda(cudaMemcpyAsync(dev, host, size_t(n) * sizeof(int32_t),
                                     cudaMemcpyHostToDevice, stream));
}

}  // extern "C"
