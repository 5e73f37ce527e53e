// Native step pipeline: a stream of steps under fixed limits, run end to end from host
// buffers with the per-step host work in one call.
//
// A serving loop runs the same step over and over: plan it on the host, upload its metadata
// and the new tokens' q / k / v, write the new K/V into the pools, attend, read the output
// back. Two slots (each with its own device metadata, q / k_new / v_new / out buffers,
// workspace, pinned host metadata and a CUDA graph of its KV write + attention, captured
// once) take alternate steps, and three streams carry the uploads, the kernels and the
// read-back, so that one step's planning and copies overlap the kernels of the step before
// it; the kernels themselves run in submission order on one stream, since every step writes
// and reads the same pools. What is run per step is exactly paged_kv_write (or its fp8 form)
// followed by paged_attention_step over a plan from pa_plan_step_shared ("P3: native paged-KV
// continuous-batching sampler", Design / engine.py: one flat ragged step per engine step).
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "../../include/pagedattn.h"
#include "common.h"

using namespace pa_detail;

struct pa_pipeline {
    pa_shape shape;
    int32_t B, T, max_blocks, max_ctx, cap;
    bool fp8;
    float k_scale, v_scale;
    void* k_pool;
    void* v_pool;
    size_t meta_ints, q_bytes, kv_bytes, ws_bytes;
    // offsets (in int32) of the metadata parts: items, cu, ctx, table, slots
    size_t o_items, o_cu, o_ctx, o_table, o_slots;
    struct Slot {
        int32_t* d_meta = nullptr;
        int32_t* h_meta = nullptr;     // pinned
        void* q = nullptr;
        void* k_new = nullptr;
        void* v_new = nullptr;
        void* out = nullptr;
        void* ws = nullptr;
        int32_t* err = nullptr;
        cudaGraphExec_t exec = nullptr;
        cudaEvent_t inputs = nullptr, computed = nullptr, done = nullptr;
        bool pending = false;
        int32_t n_planned = 0, table_cols = 0;
    } slot[2];
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    int64_t submitted = 0;
};

namespace {

int32_t run_step(pa_pipeline* p, pa_pipeline::Slot& s, cudaStream_t st) {
    const int32_t* m = s.d_meta;
    const auto* items = reinterpret_cast<const pa_work_item*>(m + p->o_items);
    int32_t r;
    if (p->fp8) {
        r = paged_kv_write_fp8(s.k_new, s.v_new, m + p->o_slots, p->T, p->k_pool, p->v_pool,
                               p->k_scale, p->v_scale, &p->shape, s.err, st);
        if (r) return r;
        return paged_attention_step_fp8(s.q, p->k_pool, p->v_pool, m + p->o_table, p->max_blocks,
                                        m + p->o_cu, m + p->o_ctx, p->B, p->T, p->max_ctx, items,
                                        p->cap, p->k_scale, p->v_scale, s.ws, p->ws_bytes, s.out,
                                        &p->shape, s.err, st);
    }
    r = paged_kv_write(s.k_new, s.v_new, m + p->o_slots, p->T, p->k_pool, p->v_pool, &p->shape,
                       s.err, st);
    if (r) return r;
    return paged_attention_step(s.q, p->k_pool, p->v_pool, m + p->o_table, p->max_blocks,
                                m + p->o_cu, m + p->o_ctx, p->B, p->T, p->max_ctx, items, p->cap,
                                s.ws, p->ws_bytes, s.out, &p->shape, s.err, st);
}

void release(pa_pipeline* p) {
    if (!p) return;
    for (auto& s : p->slot) {
        if (s.pending && s.done) cudaEventSynchronize(s.done);
        if (s.exec) cudaGraphExecDestroy(s.exec);
        for (cudaEvent_t e : {s.inputs, s.computed, s.done})
            if (e) cudaEventDestroy(e);
        for (void* d : {static_cast<void*>(s.d_meta), s.q, s.k_new, s.v_new, s.out, s.ws,
                        static_cast<void*>(s.err)})
            if (d) cudaFree(d);
        if (s.h_meta) cudaFreeHost(s.h_meta);
    }
    for (cudaStream_t st : {p->h2d, p->comp, p->d2h})
        if (st) cudaStreamDestroy(st);
    delete p;
}

}  // namespace

extern "C" int32_t pa_pipeline_create(const pa_shape* shape, int32_t B, int32_t T,
                                      int32_t max_blocks, int32_t max_ctx, void* k_pool,
                                      void* v_pool, int32_t fp8, float k_scale, float v_scale,
                                      pa_pipeline** out) {
    if (!out) return PA_ERR_INVALID;
    *out = nullptr;
    int32_t st = check_shape(shape);
    if (st) return st;
    if (B < 1 || T < 1 || max_blocks < 1 || max_ctx < 1 || !k_pool || !v_pool)
        return PA_ERR_INVALID;
    if (fp8 && (!(k_scale > 0.f) || !(v_scale > 0.f) || !(k_scale < INFINITY) ||
                !(v_scale < INFINITY)))
        return PA_ERR_INVALID;
    const int64_t cap = pa_plan_max_items_shared(shape, B, T, max_ctx);
    constexpr int64_t kItemInts = sizeof(pa_work_item) / 4;
    if (cap <= 0 || cap > INT32_MAX / kItemInts) return PA_ERR_INVALID;
    auto* p = new pa_pipeline();
    p->shape = *shape;
    p->B = B;
    p->T = T;
    p->max_blocks = max_blocks;
    p->max_ctx = max_ctx;
    p->cap = int32_t(cap);
    p->fp8 = fp8 != 0;
    p->k_scale = fp8 ? k_scale : 1.f;
    p->v_scale = fp8 ? v_scale : 1.f;
    p->k_pool = k_pool;
    p->v_pool = v_pool;
    p->o_items = 0;
    p->o_cu = size_t(cap) * size_t(kItemInts);
    p->o_ctx = p->o_cu + size_t(B) + 1;
    p->o_table = p->o_ctx + size_t(B);
    p->o_slots = p->o_table + size_t(B) * size_t(max_blocks);
    p->meta_ints = p->o_slots + size_t(T);
    const int D = shape->head_dim;
    p->q_bytes = size_t(T) * shape->num_q_heads * D * 2;
    p->kv_bytes = size_t(T) * shape->num_kv_heads * D * 2;
    p->ws_bytes = pa_workspace_bytes(shape, T, max_ctx);
    const auto fail = [&](cudaError_t e) {
        const int32_t r = note_cuda(e);
        release(p);
        return r;
    };
    cudaError_t e;
    for (cudaStream_t* sp : {&p->h2d, &p->comp, &p->d2h})
        if ((e = cudaStreamCreateWithFlags(sp, cudaStreamNonBlocking)) != cudaSuccess)
            return fail(e);
    for (auto& s : p->slot) {
        if ((e = cudaMalloc(&s.d_meta, p->meta_ints * 4)) != cudaSuccess ||
            (e = cudaMallocHost(&s.h_meta, p->meta_ints * 4)) != cudaSuccess ||
            (e = cudaMalloc(&s.q, p->q_bytes)) != cudaSuccess ||
            (e = cudaMalloc(&s.k_new, p->kv_bytes)) != cudaSuccess ||
            (e = cudaMalloc(&s.v_new, p->kv_bytes)) != cudaSuccess ||
            (e = cudaMalloc(&s.out, p->q_bytes)) != cudaSuccess ||
            (e = cudaMalloc(&s.err, 4)) != cudaSuccess ||
            (p->ws_bytes && (e = cudaMalloc(&s.ws, p->ws_bytes)) != cudaSuccess))
            return fail(e);
        for (cudaEvent_t* ev : {&s.inputs, &s.computed, &s.done})
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess)
                return fail(e);
        // every item padding, every slot -1, the table -1: a step over this metadata writes
        // and computes nothing, which is what the warm-up and the capture below run over
        std::memset(s.h_meta, 0, p->meta_ints * 4);
        for (size_t i = p->o_table; i < p->meta_ints; ++i) s.h_meta[i] = -1;
        if ((e = cudaMemcpy(s.d_meta, s.h_meta, p->meta_ints * 4, cudaMemcpyHostToDevice)) !=
                cudaSuccess ||
            (e = cudaMemset(s.q, 0, p->q_bytes)) != cudaSuccess ||
            (e = cudaMemset(s.k_new, 0, p->kv_bytes)) != cudaSuccess ||
            (e = cudaMemset(s.v_new, 0, p->kv_bytes)) != cudaSuccess ||
            (e = cudaMemset(s.err, 0, 4)) != cudaSuccess)
            return fail(e);
        // warm-up outside the capture, then the capture of the same calls
        if ((st = run_step(p, s, p->comp))) {
            release(p);
            return st;
        }
        if ((e = cudaStreamSynchronize(p->comp)) != cudaSuccess) return fail(e);
        if ((e = cudaStreamBeginCapture(p->comp, cudaStreamCaptureModeThreadLocal)) != cudaSuccess)
            return fail(e);
        st = run_step(p, s, p->comp);
        cudaGraph_t graph = nullptr;
        e = cudaStreamEndCapture(p->comp, &graph);
        if (st || e != cudaSuccess) {
            if (graph) cudaGraphDestroy(graph);
            if (st) {
                release(p);
                return st;
            }
            return fail(e);
        }
        e = cudaGraphInstantiate(&s.exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) return fail(e);
    }
    *out = p;
    return PA_OK;
}

extern "C" int32_t pa_pipeline_destroy(pa_pipeline* p) {
    release(p);
    return PA_OK;
}

extern "C" int64_t pa_pipeline_meta_bytes(const pa_pipeline* p) {
    return p ? int64_t(p->meta_ints) * 4 : -1;
}

extern "C" int32_t pa_pipeline_submit(pa_pipeline* p, const int32_t* cu_seqlens_q,
                                      const int32_t* ctx_lens, const int32_t* block_table,
                                      int32_t table_cols, const void* h_q, const void* h_k_new,
                                      const void* h_v_new, void* h_out, int32_t* slot_out) {
    if (!p || !cu_seqlens_q || !ctx_lens || !block_table || !h_q || !h_k_new || !h_v_new ||
        !h_out || table_cols < 1 || table_cols > p->max_blocks)
        return PA_ERR_INVALID;
    int32_t st = check_step_meta(p->B, cu_seqlens_q, ctx_lens);
    if (st) return st;
    if (cu_seqlens_q[p->B] != p->T) return PA_ERR_INVALID;
    for (int32_t i = 0; i < p->B; ++i)
        if (ctx_lens[i] > p->max_ctx) return PA_ERR_INVALID;
    const int which = int(p->submitted & 1);
    pa_pipeline::Slot& s = p->slot[which];
    cudaError_t e;
    // the slot's previous step has left its buffers (its output is on the host)
    if (s.pending && (e = cudaEventSynchronize(s.done)) != cudaSuccess) return note_cuda(e);
    s.pending = false;
    int32_t* h = s.h_meta;
    // the host metadata: table (row stride max_blocks, -1 past the caller's columns), slots,
    // cu, ctx and the plan, padded with n_q == 0 items past its end
    int32_t* tab = h + p->o_table;
    for (int32_t b = 0; b < p->B; ++b) {
        std::memcpy(tab + int64_t(b) * p->max_blocks, block_table + int64_t(b) * table_cols,
                    size_t(table_cols) * 4);
        for (int32_t c = table_cols; c < s.table_cols; ++c) tab[int64_t(b) * p->max_blocks + c] = -1;
    }
    s.table_cols = table_cols;
    if ((st = pa_compute_slots(&p->shape, tab, p->B, p->max_blocks, cu_seqlens_q, ctx_lens,
                               h + p->o_slots)))
        return st;
    std::memcpy(h + p->o_cu, cu_seqlens_q, size_t(p->B + 1) * 4);
    std::memcpy(h + p->o_ctx, ctx_lens, size_t(p->B) * 4);
    auto* items = reinterpret_cast<pa_work_item*>(h + p->o_items);
    int32_t n = 0;
    if ((st = pa_plan_step_shared(&p->shape, p->B, cu_seqlens_q, ctx_lens, tab, p->max_blocks, items,
                                  p->cap, &n)))
        return st;
    if (n < s.n_planned) std::memset(items + n, 0, size_t(s.n_planned - n) * sizeof(pa_work_item));
    s.n_planned = n;
    // uploads, kernels, read-back
    if ((e = cudaMemcpyAsync(s.d_meta, h, p->meta_ints * 4, cudaMemcpyHostToDevice, p->h2d)) ||
        (e = cudaMemcpyAsync(s.q, h_q, p->q_bytes, cudaMemcpyHostToDevice, p->h2d)) ||
        (e = cudaMemcpyAsync(s.k_new, h_k_new, p->kv_bytes, cudaMemcpyHostToDevice, p->h2d)) ||
        (e = cudaMemcpyAsync(s.v_new, h_v_new, p->kv_bytes, cudaMemcpyHostToDevice, p->h2d)) ||
        (e = cudaEventRecord(s.inputs, p->h2d)) ||
        (e = cudaStreamWaitEvent(p->comp, s.inputs, 0)) ||
        (e = cudaGraphLaunch(s.exec, p->comp)) ||
        (e = cudaEventRecord(s.computed, p->comp)) ||
        (e = cudaStreamWaitEvent(p->d2h, s.computed, 0)) ||
        (e = cudaMemcpyAsync(h_out, s.out, p->q_bytes, cudaMemcpyDeviceToHost, p->d2h)) ||
        (e = cudaEventRecord(s.done, p->d2h)))
        return note_cuda(e);
    s.pending = true;
    ++p->submitted;
    if (slot_out) *slot_out = which;
    return PA_OK;
}

extern "C" int32_t pa_pipeline_wait(pa_pipeline* p, int32_t slot) {
    if (!p || slot < 0 || slot > 1) return PA_ERR_INVALID;
    pa_pipeline::Slot& s = p->slot[slot];
    if (!s.pending) return PA_OK;
    const cudaError_t e = cudaEventSynchronize(s.done);
    if (e != cudaSuccess) return note_cuda(e);
    s.pending = false;
    return PA_OK;
}

extern "C" int32_t pa_pipeline_device_error(pa_pipeline* p, int32_t* err) {
    if (!p || !err) return PA_ERR_INVALID;
    *err = 0;
    for (auto& s : p->slot) {
        if (s.pending && s.done) {
            const cudaError_t e = cudaEventSynchronize(s.done);
            if (e != cudaSuccess) return note_cuda(e);
            s.pending = false;
        }
        int32_t v = 0;
        const cudaError_t e = cudaMemcpy(&v, s.err, 4, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return note_cuda(e);
        *err |= v;
    }
    return PA_OK;
}
