// KV-write scatter: the copy-free append of "P3: native paged-KV continuous-batching sampler",
// Design / paged.py ("write scatters into (block, offset) in place").
//
// One CTA per new token. A token's K row and V row are each Hkv*D bf16 = Hkv*D*2 bytes,
// contiguous in the source and in the destination slot, so the copy is a pair of dense
// 16-byte-vector streams. HBM-bound; the bytes are copied unchanged.
#include <cuda_runtime.h>

#include "common.h"

using namespace pa_detail;

namespace {

__global__ void __launch_bounds__(128) kv_write_kernel(const uint4* __restrict__ k_new,
                                                       const uint4* __restrict__ v_new,
                                                       const int32_t* __restrict__ slots,
                                                       uint4* __restrict__ k_pool,
                                                       uint4* __restrict__ v_pool,
                                                       int32_t row_vecs, int64_t num_slots,
                                                       int32_t* err) {
    // the attention kernel that follows on the stream may launch now: it waits for this
    // grid to complete before it reads the pools
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t t = blockIdx.x;
    const int32_t slot = slots[t];
    if (slot < 0) return;                         // "no write" marker
    if (slot >= num_slots) {
        if (threadIdx.x == 0 && err) atomicOr(err, PA_DEVERR_SLOT);
        return;
    }
    const uint4* ks = k_new + t * row_vecs;
    const uint4* vs = v_new + t * row_vecs;
    uint4* kd = k_pool + int64_t(slot) * row_vecs;
    uint4* vd = v_pool + int64_t(slot) * row_vecs;
    for (int32_t i = threadIdx.x; i < row_vecs; i += blockDim.x) {
        const uint4 a = __ldg(ks + i);
        const uint4 b = __ldg(vs + i);
        kd[i] = a;
        vd[i] = b;
    }
}

// Copy-on-write block copies: CTA k copies block pairs[2k] to block pairs[2k + 1] in both
// pools (block_vecs 16-byte vectors per block and pool). A pair with an id outside the pool
// or equal ids is skipped and raises PA_DEVERR_BLOCK.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const int32_t* __restrict__ pairs,
                                                          uint4* __restrict__ k_pool,
                                                          uint4* __restrict__ v_pool,
                                                          int32_t block_vecs, int32_t num_blocks,
                                                          int32_t* err) {
    const int32_t src = pairs[2 * blockIdx.x];
    const int32_t dst = pairs[2 * blockIdx.x + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks || src == dst) {
        if (threadIdx.x == 0 && err) atomicOr(err, PA_DEVERR_BLOCK);
        return;
    }
    const uint4* ks = k_pool + int64_t(src) * block_vecs;
    const uint4* vs = v_pool + int64_t(src) * block_vecs;
    uint4* kd = k_pool + int64_t(dst) * block_vecs;
    uint4* vd = v_pool + int64_t(dst) * block_vecs;
    for (int32_t i = threadIdx.x; i < block_vecs; i += blockDim.x) {
        const uint4 a = ks[i];
        const uint4 b = vs[i];
        kd[i] = a;
        vd[i] = b;
    }
}

}  // namespace

extern "C" int32_t paged_copy_blocks(const int32_t* pairs, int32_t n_pairs, void* k_pool,
                                     void* v_pool, const pa_shape* shape, int32_t* err_flag,
                                     pa_stream_t stream) {
    int32_t st = check_shape(shape);
    if (st) return st;
    if (n_pairs < 0) return PA_ERR_INVALID;
    if (n_pairs == 0) return PA_OK;
    if (!pairs || !k_pool || !v_pool) return PA_ERR_INVALID;
    const int64_t block_elems =
        int64_t(shape->block_size) * shape->num_kv_heads * shape->head_dim;
    if (block_elems % 8) return PA_ERR_SHAPE;
    const auto aligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    if (!aligned(k_pool) || !aligned(v_pool)) return PA_ERR_INVALID;
    copy_blocks_kernel<<<n_pairs, 256, 0, stream>>>(pairs, static_cast<uint4*>(k_pool),
                                                    static_cast<uint4*>(v_pool),
                                                    int32_t(block_elems / 8), shape->num_blocks,
                                                    err_flag);
    return note_cuda(cudaGetLastError());
}

extern "C" int32_t paged_kv_write(const void* k_new, const void* v_new,
                                  const int32_t* slot_mapping, int32_t T, void* k_pool,
                                  void* v_pool, const pa_shape* shape, int32_t* err_flag,
                                  pa_stream_t stream) {
    int32_t st = check_shape(shape);
    if (st) return st;
    if (T < 0) return PA_ERR_INVALID;
    if (T == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool) return PA_ERR_INVALID;
    const int64_t row_elems = int64_t(shape->num_kv_heads) * shape->head_dim;
    if (row_elems % 8) return PA_ERR_SHAPE;
    const auto aligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    if (!aligned(k_new) || !aligned(v_new) || !aligned(k_pool) || !aligned(v_pool))
        return PA_ERR_INVALID;
    const int64_t num_slots = int64_t(shape->num_blocks) * shape->block_size;
    kv_write_kernel<<<T, 128, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), int32_t(row_elems / 8),
        num_slots, err_flag);
    return note_cuda(cudaGetLastError());
}
