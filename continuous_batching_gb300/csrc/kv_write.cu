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

// FP8 KV write ("P3: native paged-KV continuous-batching sampler", Review, kv_dtype item: an
// fp8 cache needs per-tensor scales; "Finish RL Training Faster: Bitwise-Consistent, ...",
// 4.2: prefill and decode share the write path): code = e4m3(x / s), the division in fp32
// with IEEE rounding, then round to nearest (ties to even) with saturation at +-448.
// Two bf16 -> two codes; lo lands in the lower byte (the lower address).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// 8 bf16 (a uint4) / s -> 8 codes (two words)
__device__ __forceinline__ uint2 quantize8(uint4 v, float s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        h[i] = e4m3x2(__fdiv_rn(__uint_as_float(w[i] << 16), s),
                      __fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), s));
    return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

// One CTA per new token; a thread turns 16 bf16 values (two 16-byte loads) into 16 codes
// (one 16-byte store) of the token's K row and of its V row.
__global__ void __launch_bounds__(128) kv_write_fp8_kernel(const uint4* __restrict__ k_new,
                                                           const uint4* __restrict__ v_new,
                                                           const int32_t* __restrict__ slots,
                                                           uint4* __restrict__ k_pool,
                                                           uint4* __restrict__ v_pool,
                                                           int32_t row_chunks, int64_t num_slots,
                                                           float k_scale, float v_scale,
                                                           int32_t* err) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t t = blockIdx.x;
    const int32_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (threadIdx.x == 0 && err) atomicOr(err, PA_DEVERR_SLOT);
        return;
    }
    const uint4* ks = k_new + t * 2 * row_chunks;
    const uint4* vs = v_new + t * 2 * row_chunks;
    uint4* kd = k_pool + int64_t(slot) * row_chunks;
    uint4* vd = v_pool + int64_t(slot) * row_chunks;
    for (int32_t i = threadIdx.x; i < row_chunks; i += blockDim.x) {
        const uint2 k0 = quantize8(__ldg(ks + 2 * i), k_scale);
        const uint2 k1 = quantize8(__ldg(ks + 2 * i + 1), k_scale);
        const uint2 v0 = quantize8(__ldg(vs + 2 * i), v_scale);
        const uint2 v1 = quantize8(__ldg(vs + 2 * i + 1), v_scale);
        kd[i] = make_uint4(k0.x, k0.y, k1.x, k1.y);
        vd[i] = make_uint4(v0.x, v0.y, v1.x, v1.y);
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

extern "C" int32_t paged_kv_write_fp8(const void* k_new, const void* v_new,
                                      const int32_t* slot_mapping, int32_t T, void* k_pool,
                                      void* v_pool, float k_scale, float v_scale,
                                      const pa_shape* shape, int32_t* err_flag,
                                      pa_stream_t stream) {
    int32_t st = check_shape(shape);
    if (st) return st;
    if (T < 0 || !(k_scale > 0.f) || !(v_scale > 0.f) || !(k_scale < INFINITY) ||
        !(v_scale < INFINITY))
        return PA_ERR_INVALID;
    if (T == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool) return PA_ERR_INVALID;
    const int64_t row_elems = int64_t(shape->num_kv_heads) * shape->head_dim;
    if (row_elems % 16) return PA_ERR_SHAPE;
    const auto aligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    if (!aligned(k_new) || !aligned(v_new) || !aligned(k_pool) || !aligned(v_pool))
        return PA_ERR_INVALID;
    const int64_t num_slots = int64_t(shape->num_blocks) * shape->block_size;
    kv_write_fp8_kernel<<<T, 128, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), int32_t(row_elems / 16),
        num_slots, k_scale, v_scale, err_flag);
    return note_cuda(cudaGetLastError());
}
