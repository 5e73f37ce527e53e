// Paged attention for one flat ragged step on sm_103a: one tile routine for every query row.
//
// What it computes: "P3: native paged-KV continuous-batching sampler", Design / paged.py
// ('row' mode: each query row attends exactly its own keys; kernel contract: q, K/V cache
// blocks, block tables, cu_seqlens_q, ctx_lens; fixed KV split per context length, no
// atomics) and Design / engine.py (decode rows and chunked-prefill segments in one flat
// ragged step). Why one routine for both phases: "Finish RL Training Faster: Bitwise-
// Consistent, High-Performance, Agent-Driven", section 2 (phase consistency) and 4.2 (decode
// routed through the prefill read path).
//
// Work item = (sequence, KV head, tile of up to 128/g query tokens, KV split). The M = 128
// rows of every MMA are (token, head-in-group) pairs of one KV head, so K/V tiles are shared
// by the g query heads of a group. A decode item simply has one token (g valid rows). Every
// row runs the same instruction sequence whatever the item holds:
//   S  = Q K^T    tcgen05.mma kind::f16, M 128 x N 128 keys x K D, fp32 in TMEM
//   softmax       fp32 online softmax over 128-key tiles aligned to absolute key positions;
//                 a row is spread over 4 threads (tcgen05.ld 16x256b); fixed reduction order
//   O += P V      tcgen05.mma, M 128 x N D x K 128 keys, P rounded to bf16 in shared memory
// A tensor-core output element depends only on its own row of A and column of B, so a row's
// bits do not depend on the other rows of the tile; the fixed splits
// [s*1024, (s+1)*1024) and the ascending-order combine make them independent of the batch.
//
// Warp roles (192 threads): warps 0-3 softmax / rescale / epilogue, warp 4 TMA producer,
// warp 5 MMA issuer and TMEM owner. K/V blocks arrive by TMA (one box per block and 64-column
// half, 128-byte swizzle) into a 2-stage ring; every wait on an mbarrier is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "common.h"
#include "tmem_ldst.h"

using namespace pa_detail;

namespace {

constexpr int kRows = PA_ROWS;
constexpr int kTileKeys = PA_TILE_KEYS;
constexpr int kSplit = PA_SPLIT_TOKENS;
constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;                 // S: columns [0,128), O: [128, 128 + D)
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // one second per wait

static_assert(kSplit % kTileKeys == 0, "splits are whole tiles");

template <int D>
struct Layout {
    static constexpr int kChunks = D / 64;                  // 128-byte column chunks of a row
    static constexpr int kQHalf = kRows * 128;              // bytes of one chunk column of Q
    static constexpr int kKVHalf = kTileKeys * 128;
    static constexpr int kQ = 0;
    static constexpr int kP = kQ + kChunks * kQHalf;        // P: 128 keys = 2 chunks
    static constexpr int kK = kP + 2 * kRows * 128;
    static constexpr int kKVStage = kChunks * kKVHalf;
    static constexpr int kV = kK + kStages * kKVStage;
    static constexpr int kBar = kV + kStages * kKVStage;
    static constexpr int kBytes = kBar + 256;
    static constexpr int kAlloc = kBytes + 1024;            // room to align the base to 1024
};

// mbarrier slots (8 bytes each) at Layout::kBar
enum Bar { kKVFull0 = 0, kKVFull1, kKVEmpty0, kKVEmpty1, kSFull, kPFull, kOFull, kQFull, kDrain,
           kNumBars };
constexpr int kHolderOff = 8 * kNumBars;          // TMEM address written by tcgen05.alloc
constexpr int kAbortOff = kHolderOff + 4;

struct Params {
    const __nv_bfloat16* q;
    const int32_t* block_table;
    const int32_t* cu;
    const int32_t* ctx;
    const pa_work_item* items;
    float* ws_acc;      // [T][max_splits][Hq][D]
    float* ws_ml;       // [T][max_splits][Hq][2]
    __nv_bfloat16* out;
    int32_t* err;
    int32_t B, T, max_blocks, max_splits, Hq, Hkv, g, bs, num_blocks;
    float c;            // log2(e) / sqrt(D): softmax works in base 2 on raw scores
};

// ----------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with the given parity. Gives up when another role has set
// the CTA's abort word or after kWaitLimitNs; then sets the abort word and returns false.
__device__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_word) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_word) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort_word = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulator).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and B bf16 (bits 7-9,
// 10-12 = 1), A K-major, B K-major or MN-major (bit 16), N >> 3 at bits 17-22, M >> 4 at
// bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor: start address >> 4 (bits 0-13), leading-dimension byte
// offset >> 4 (16-29), stride-dimension byte offset >> 4 (32-45), descriptor version 1
// (bit 46), 128-byte swizzle (layout type 2, bits 61-63). Operand tiles sit at 1024-byte
// aligned addresses in rows of 128 bytes, 8-row swizzle atoms.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((addr & 0x3FFFF) >> 4) | (uint64_t((lbo >> 4) & 0x3FFF) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFF) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// 2^x on the special-function unit (ex2.approx, flush-to-zero). Every place that takes an
// exponential in this library calls this one helper, so all of them round the same way.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
}

// Offset of 16-byte chunk `chunk` (0..7) of row `row` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return uint32_t(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// --------------------------------------------------------------- the tile routine

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    paged_attn_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const Params p) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t bars = sb + L::kBar;
    volatile int* abort_word = reinterpret_cast<volatile int*>(smem + L::kBar + kAbortOff);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    pa_work_item it = p.items[blockIdx.x];
    // The item and the metadata it points at are device data: check them before use. A bad
    // item does no work (n_tiles = 0) and raises PA_DEVERR_META.
    bool good = it.seq >= 0 && it.seq < p.B && it.kv_head >= 0 && it.kv_head < p.Hkv &&
                it.n_q >= 1 && it.n_q * p.g <= kRows && it.split >= 0 && it.q_start >= 0 &&
                it.q_start + it.n_q <= p.T;
    const int seq = good ? it.seq : 0;
    const int ctx_s = good ? p.ctx[seq] : 0;
    const int cu0 = good ? p.cu[seq] : 0;
    const int cu1 = good ? p.cu[seq + 1] : 0;
    good = good && cu0 <= it.q_start && it.q_start + it.n_q <= cu1 && cu1 - cu0 <= ctx_s &&
           (int64_t(ctx_s) + p.bs - 1) / p.bs <= p.max_blocks;
    const int pos0 = ctx_s - cu1 + it.q_start;              // position of the item's first row
    const int p_max = pos0 + it.n_q - 1;
    const int k_begin = it.split * kSplit;
    good = good && k_begin <= p_max && (p_max < kSplit || p_max / kSplit < p.max_splits);
    const int k_end = min(k_begin + kSplit, p_max + 1);
    const int n_tiles = good ? (k_end - k_begin + kTileKeys - 1) / kTileKeys : 0;
    const int rows_valid = good ? it.n_q * p.g : 0;
    if (!good && threadIdx.x == 0 && p.err) atomicOr(p.err, PA_DEVERR_META);

    if (threadIdx.x == 0) {
        for (int b = 0; b < kNumBars; ++b)
            mbar_init(bars + 8 * b, (b == kPFull || b == kQFull) ? 128 : 1);
        *abort_word = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         bars + kHolderOff),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kBar + kHolderOff);
    const uint32_t tm_s = tmem;
    const uint32_t tm_o = tmem + 128;

    if (warp == 4) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n_tiles > 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
            const int32_t* trow = p.block_table + int64_t(seq) * p.max_blocks;
            const int kvh = it.kv_head;
            int issued = 0;
            for (int jt = 0; jt < n_tiles; ++jt) {
                const int st = jt & 1;
                if (jt >= 2 && !wait_bounded(bars + 8 * (kKVEmpty0 + st), ((jt >> 1) - 1) & 1,
                                             abort_word))
                    break;
                const int kb = k_begin + jt * kTileKeys;
                const int key_hi = min(kb + kTileKeys, ctx_s);       // real keys end at ctx
                const int nblk = (key_hi - kb + p.bs - 1) / p.bs;
                const uint32_t bar = bars + 8 * (kKVFull0 + st);
                mbar_expect_tx(bar, uint32_t(nblk) * p.bs * 128 * L::kChunks * 2);
                const uint32_t dk = sb + L::kK + st * L::kKVStage;
                const uint32_t dv = sb + L::kV + st * L::kKVStage;
                for (int b = 0; b < nblk; ++b) {
                    int phys = trow[kb / p.bs + b];
                    if (phys < 0 || phys >= p.num_blocks) {
                        // out of range: the box lands outside the tensor and reads as zeros
                        if (p.err) atomicOr(p.err, PA_DEVERR_BLOCK);
                        phys = -1;
                    }
                    const int z = phys * p.bs;
                    for (int h = 0; h < L::kChunks; ++h) {
                        const uint32_t off = h * L::kKVHalf + b * p.bs * 128;
                        tma_load_3d(dk + off, &tm_k, bar, 64 * h, kvh, z);
                        tma_load_3d(dv + off, &tm_v, bar, 64 * h, kvh, z);
                    }
                }
                ++issued;
            }
            // never leave with copies in flight into this CTA's shared memory
            for (int jt = max(0, issued - 2); jt < issued; ++jt)
                wait_bounded(bars + 8 * (kKVFull0 + (jt & 1)), (jt >> 1) & 1, abort_word);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t idesc_s = make_idesc(kRows, kTileKeys, false);
            constexpr uint32_t idesc_o = make_idesc(kRows, D, true);
            const auto issue_s = [&](int jt) {
                const uint32_t kbase = sb + L::kK + (jt & 1) * L::kKVStage;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t qa = sb + L::kQ + (k >> 2) * L::kQHalf + (k & 3) * 32;
                    const uint32_t ka = kbase + (k >> 2) * L::kKVHalf + (k & 3) * 32;
                    umma_bf16(tm_s, make_sdesc(qa, 16, 1024), make_sdesc(ka, 16, 1024), idesc_s,
                              k > 0);
                }
            };
            const auto issue_pv = [&](int jt) {
                const uint32_t vbase = sb + L::kV + (jt & 1) * L::kKVStage;
#pragma unroll
                for (int k = 0; k < kTileKeys / 16; ++k) {
                    const uint32_t pa = sb + L::kP + (k >> 2) * (kRows * 128) + (k & 3) * 32;
                    const uint32_t va = vbase + k * 16 * 128;
                    umma_bf16(tm_o, make_sdesc(pa, 16, 1024), make_sdesc(va, L::kKVHalf, 1024),
                              idesc_o, (jt > 0 || k > 0) ? 1u : 0u);
                }
            };
            bool ok = wait_bounded(bars + 8 * kQFull, 0, abort_word);
            tc_fence_after();
            for (int jt = 0; ok && jt < n_tiles; ++jt) {
                if (jt > 0) {
                    if (!(ok = wait_bounded(bars + 8 * kPFull, (jt - 1) & 1, abort_word))) break;
                    tc_fence_after();
                    issue_pv(jt - 1);
                    tc_commit(bars + 8 * (kKVEmpty0 + ((jt - 1) & 1)));
                }
                if (!(ok = wait_bounded(bars + 8 * (kKVFull0 + (jt & 1)), (jt >> 1) & 1,
                                        abort_word)))
                    break;
                tc_fence_after();
                issue_s(jt);
                tc_commit(bars + 8 * kSFull);
            }
            if (ok && wait_bounded(bars + 8 * kPFull, (n_tiles - 1) & 1, abort_word)) {
                tc_fence_after();
                issue_pv(n_tiles - 1);
                tc_commit(bars + 8 * (kKVEmpty0 + ((n_tiles - 1) & 1)));
                tc_commit(bars + 8 * kOFull);
            }
            // drain: every MMA this thread issued has finished before TMEM is released
            tc_commit(bars + 8 * kDrain);
            wait_bounded(bars + 8 * kDrain, 0, abort_word);
        }
    } else {
        // ------------------------------------------------------------ softmax warps 0-3
        const int tid = threadIdx.x;              // 0..127
        // zero P, then stage Q rows (token-major, head-in-group minor) in the swizzled layout
        for (int i = tid; i < 2 * kRows * 8; i += 128) st_shared_zero16(sb + L::kP + i * 16);
        constexpr int kRowChunks = D / 8;          // 16-byte chunks per row
        for (int i = tid; i < kRows * kRowChunks; i += 128) {
            const int r = i / kRowChunks;
            const int ch = i % kRowChunks;
            const uint32_t dst = sb + L::kQ + (ch >> 3) * L::kQHalf + swz(r, ch & 7);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < rows_valid) {
                const int tok = it.q_start + r / p.g;
                const int head = it.kv_head * p.g + r % p.g;
                v = __ldg(reinterpret_cast<const uint4*>(p.q + (int64_t(tok) * p.Hq + head) * D) + ch);
            }
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y),
                         "r"(v.z), "r"(v.w)
                         : "memory");
        }
        fence_proxy_async();
        mbar_arrive(bars + 8 * kQFull);            // all 128 softmax threads arrive

        const int q4 = lane & 3;
        const int rs = lane >> 2;
        bool half_on[2];
        int pos[2][2];
        float m_run[2][2], l_run[2][2], alpha[2][2];
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            half_on[hb] = (32 * warp + 16 * hb) < rows_valid;
#pragma unroll
            for (int sr = 0; sr < 2; ++sr) {
                const int row = 32 * warp + 16 * hb + rs + 8 * sr;
                pos[hb][sr] = row < rows_valid ? pos0 + row / p.g : -1;
                m_run[hb][sr] = -INFINITY;
                l_run[hb][sr] = 0.f;
                alpha[hb][sr] = 1.f;
            }
        }
        const float c = p.c;
        bool ok = true;
        for (int jt = 0; jt < n_tiles; ++jt) {
            if (!(ok = wait_bounded(bars + 8 * kSFull, jt & 1, abort_word))) break;
            tc_fence_after();
            const int kb = k_begin + jt * kTileKeys;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                if (!half_on[hb]) continue;
                uint32_t r[64];
                tmem_ld_16x256b_x16(tm_s + (uint32_t(32 * warp + 16 * hb) << 16), r);
                tmem_wait_ld();
#pragma unroll
                for (int sr = 0; sr < 2; ++sr) {
                    const int row = 32 * warp + 16 * hb + rs + 8 * sr;
                    const int pr = pos[hb][sr];
                    float sv[32];
                    float mx = -INFINITY;
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int key = kb + 8 * cc + 2 * q4 + e;
                            const float s = key <= pr ? __uint_as_float(r[4 * cc + 2 * sr + e])
                                                      : -INFINITY;
                            sv[2 * cc + e] = s;
                            mx = fmaxf(mx, s);
                        }
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    const float m_new = fmaxf(m_run[hb][sr], mx);
                    const float m_use = m_new == -INFINITY ? 0.f : m_new;
                    const float a = m_run[hb][sr] == m_use
                                        ? 1.f
                                        : ex2(__fmul_rn(__fsub_rn(m_run[hb][sr], m_use), c));
                    const float nmc = __fmul_rn(-m_use, c);
                    float sum = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        sv[i] = ex2(__fmaf_rn(sv[i], c, nmc));
                        sum = __fadd_rn(sum, sv[i]);
                    }
                    sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 1));
                    sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 2));
                    l_run[hb][sr] = __fadd_rn(__fmul_rn(l_run[hb][sr], a), sum);
                    m_run[hb][sr] = m_new;
                    alpha[hb][sr] = a;
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc) {
                        const uint32_t addr = sb + L::kP + (cc >> 3) * (kRows * 128) +
                                              swz(row, cc & 7) + 4 * q4;
                        st_shared_u32(addr, pack_bf16(sv[2 * cc], sv[2 * cc + 1]));
                    }
                }
            }
            // keys at or beyond ctx are stale or never loaded: give them zero values so that
            // their (zero) probabilities contribute exact zeros
            if (kb + kTileKeys > ctx_s) {
                const int r0 = max(ctx_s - kb, 0);
                const int nrow = kTileKeys - r0;
                const uint32_t vb = sb + L::kV + (jt & 1) * L::kKVStage;
                for (int i = tid; i < nrow * 8 * L::kChunks; i += 128) {
                    const int h = i / (nrow * 8);
                    const int rem = i % (nrow * 8);
                    st_shared_zero16(vb + h * L::kKVHalf + (r0 + rem / 8) * 128 + (rem % 8) * 16);
                }
            }
            if (jt > 0) {
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    if (!half_on[hb]) continue;
                    const bool need = alpha[hb][0] != 1.f || alpha[hb][1] != 1.f;
                    if (!__any_sync(0xffffffffu, need)) continue;
                    const uint32_t ta = tm_o + (uint32_t(32 * warp + 16 * hb) << 16);
                    if constexpr (D == 128) {
                        uint32_t o[64];
                        tmem_ld_16x256b_x16(ta, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int cc = 0; cc < 16; ++cc)
#pragma unroll
                            for (int sr = 0; sr < 2; ++sr)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const int k = 4 * cc + 2 * sr + e;
                                    o[k] = __float_as_uint(
                                        __fmul_rn(__uint_as_float(o[k]), alpha[hb][sr]));
                                }
                        tmem_st_16x256b_x16(ta, o);
                    } else {
                        uint32_t o[32];
                        tmem_ld_16x256b_x8(ta, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc)
#pragma unroll
                            for (int sr = 0; sr < 2; ++sr)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const int k = 4 * cc + 2 * sr + e;
                                    o[k] = __float_as_uint(
                                        __fmul_rn(__uint_as_float(o[k]), alpha[hb][sr]));
                                }
                        tmem_st_16x256b_x8(ta, o);
                    }
                }
                tmem_wait_st();
            }
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(bars + 8 * kPFull);        // all 128 softmax threads arrive
        }
        // ---------------------------------------------------------------- epilogue
        if (ok && n_tiles > 0 && wait_bounded(bars + 8 * kOFull, 0, abort_word)) {
            tc_fence_after();
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                if (!half_on[hb]) continue;
                const uint32_t ta = tm_o + (uint32_t(32 * warp + 16 * hb) << 16);
                uint32_t o[D / 2];
                if constexpr (D == 128) tmem_ld_16x256b_x16(ta, o);
                else tmem_ld_16x256b_x8(ta, o);
                tmem_wait_ld();
#pragma unroll
                for (int sr = 0; sr < 2; ++sr) {
                    const int row = 32 * warp + 16 * hb + rs + 8 * sr;
                    if (row >= rows_valid) continue;
                    const int pr = pos[hb][sr];
                    const int nsp = pr / kSplit + 1;
                    if (it.split >= nsp) continue;      // the row has no keys in this split
                    const int tok = it.q_start + row / p.g;
                    const int head = it.kv_head * p.g + row % p.g;
                    if (nsp == 1) {
                        const float lsum = l_run[hb][sr];
                        __nv_bfloat16* dst = p.out + (int64_t(tok) * p.Hq + head) * D;
#pragma unroll
                        for (int cc = 0; cc < D / 8; ++cc) {
                            const float x0 = __fdiv_rn(__uint_as_float(o[4 * cc + 2 * sr]), lsum);
                            const float x1 = __fdiv_rn(__uint_as_float(o[4 * cc + 2 * sr + 1]), lsum);
                            *reinterpret_cast<uint32_t*>(dst + 8 * cc + 2 * q4) = pack_bf16(x0, x1);
                        }
                    } else {
                        const int64_t slot = (int64_t(tok) * p.max_splits + it.split) * p.Hq + head;
                        float* acc = p.ws_acc + slot * D;
#pragma unroll
                        for (int cc = 0; cc < D / 8; ++cc)
                            *reinterpret_cast<float2*>(acc + 8 * cc + 2 * q4) =
                                make_float2(__uint_as_float(o[4 * cc + 2 * sr]),
                                            __uint_as_float(o[4 * cc + 2 * sr + 1]));
                        if (q4 == 0)
                            *reinterpret_cast<float2*>(p.ws_ml + slot * 2) =
                                make_float2(m_run[hb][sr], l_run[hb][sr]);
                    }
                }
            }
        }
    }
    if (*abort_word && threadIdx.x == 0 && p.err) atomicOr(p.err, PA_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------- fixed-order split combine
// For every (row, q head) whose row spans more than one split: fold the partials of splits
// 0, 1, ... in ascending order, starting from split 0's (m, l, acc) as they are:
//   M' = max(M, m_s), a = 2^((M - M') c), b = 2^((m_s - M') c),
//   L = L a + l_s b, ACC = ACC a + acc_s b;  out = bf16_rne(ACC / L).
// A row with one split is finished by the attention kernel with the same division.
template <int D>
__global__ void __launch_bounds__(128)
    combine_kernel(const float* __restrict__ ws_acc, const float* __restrict__ ws_ml,
                   const int32_t* __restrict__ cu, const int32_t* __restrict__ ctx, int32_t B,
                   int32_t T, int32_t Hq, int32_t max_splits, float c,
                   __nv_bfloat16* __restrict__ out) {
    constexpr int E = D / 32;
    const int64_t w = int64_t(blockIdx.x) * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t tok = w / Hq;
    const int head = int(w % Hq);
    if (tok >= T) return;
    int lo = 0, hi = B - 1;                     // sequence s with cu[s] <= tok < cu[s+1]
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= tok) lo = mid;
        else hi = mid - 1;
    }
    const int pos = ctx[lo] - cu[lo + 1] + int(tok);
    if (pos < 0) return;                         // inconsistent metadata: flagged by the kernel
    const int nsp = pos / kSplit + 1;
    if (nsp == 1 || nsp > max_splits) return;
    const int64_t base = tok * max_splits;
    float acc[E];
    float M, Lsum;
    {
        const int64_t slot = base * Hq + head;
        const float2 ml = *reinterpret_cast<const float2*>(ws_ml + slot * 2);
        M = ml.x;
        Lsum = ml.y;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = ws_acc[slot * D + lane * E + e];
    }
    for (int s = 1; s < nsp; ++s) {
        const int64_t slot = (base + s) * Hq + head;
        const float2 ml = *reinterpret_cast<const float2*>(ws_ml + slot * 2);
        const float mn = fmaxf(M, ml.x);
        const float fa = M == mn ? 1.f : ex2(__fmul_rn(__fsub_rn(M, mn), c));
        const float fb = ml.x == mn ? 1.f : ex2(__fmul_rn(__fsub_rn(ml.x, mn), c));
        Lsum = __fadd_rn(__fmul_rn(Lsum, fa), __fmul_rn(ml.y, fb));
#pragma unroll
        for (int e = 0; e < E; ++e)
            acc[e] = __fadd_rn(__fmul_rn(acc[e], fa),
                               __fmul_rn(ws_acc[slot * D + lane * E + e], fb));
        M = mn;
    }
    __nv_bfloat16* dst = out + (tok * Hq + head) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2)
        *reinterpret_cast<uint32_t*>(dst + e) =
            pack_bf16(__fdiv_rn(acc[e], Lsum), __fdiv_rn(acc[e + 1], Lsum));
}

// ------------------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// Pool viewed as a 3-D tensor {D, Hkv, num_blocks * block_size}; one box is one block of one
// KV head and one 64-element column chunk, 128-byte swizzled in shared memory.
int32_t make_pool_map(CUtensorMap* m, const void* pool, const pa_shape* s) {
    auto fn = encode_fn();
    if (!fn) return PA_ERR_CUDA;
    const cuuint64_t dims[3] = {cuuint64_t(s->head_dim), cuuint64_t(s->num_kv_heads),
                                cuuint64_t(s->num_blocks) * s->block_size};
    const cuuint64_t strides[2] = {cuuint64_t(s->head_dim) * 2,
                                   cuuint64_t(s->num_kv_heads) * s->head_dim * 2};
    const cuuint32_t box[3] = {64, 1, cuuint32_t(s->block_size)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

template <int D>
int32_t launch(const CUtensorMap& mk, const CUtensorMap& mv, const Params& prm, int32_t n_items,
               int32_t B, int32_t T, int32_t max_ctx, cudaStream_t stream) {
    static int attr_device = -1;          // device the shared-memory limit was raised on
    int dev = 0;
    int32_t st0 = note_cuda(cudaGetDevice(&dev));
    if (st0) return st0;
    if (attr_device != dev) {
        st0 = note_cuda(cudaFuncSetAttribute(
            paged_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<D>::kAlloc));
        if (st0) return st0;
        attr_device = dev;
    }
    paged_attn_kernel<D><<<n_items, kThreads, Layout<D>::kAlloc, stream>>>(mk, mv, prm);
    int32_t st = note_cuda(cudaGetLastError());
    if (st) return st;
    if (max_ctx > kSplit) {
        const int64_t warps = int64_t(T) * prm.Hq;
        combine_kernel<D><<<unsigned((warps + 3) / 4), 128, 0, stream>>>(
            prm.ws_acc, prm.ws_ml, prm.cu, prm.ctx, B, T, prm.Hq, prm.max_splits, prm.c, prm.out);
        st = note_cuda(cudaGetLastError());
    }
    return st;
}

}  // namespace

extern "C" int32_t paged_attention_step(const void* q, const void* k_pool, const void* v_pool,
                                        const int32_t* block_table, int32_t max_blocks,
                                        const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                                        int32_t B, int32_t T, int32_t max_ctx,
                                        const pa_work_item* items, int32_t n_items,
                                        void* workspace, size_t ws_bytes, void* out,
                                        const pa_shape* shape, int32_t* err_flag,
                                        pa_stream_t stream) {
    int32_t st = check_shape(shape);
    if (st) return st;
    if (B < 0 || T < 0 || n_items < 0 || max_ctx < 0 || max_blocks < 0) return PA_ERR_INVALID;
    if (T == 0 || n_items == 0) return PA_OK;
    if (!q || !k_pool || !v_pool || !block_table || !cu_seqlens_q || !ctx_lens || !items || !out)
        return PA_ERR_INVALID;
    if (int64_t(shape->num_blocks) * shape->block_size > INT32_MAX) return PA_ERR_SHAPE;
    const size_t need = pa_workspace_bytes(shape, T, max_ctx);
    if (max_ctx > kSplit && (!workspace || ws_bytes < need)) return PA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool) |
         reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15)
        return PA_ERR_INVALID;

    CUtensorMap mk, mv;
    if ((st = make_pool_map(&mk, k_pool, shape))) return st;
    if ((st = make_pool_map(&mv, v_pool, shape))) return st;

    const int D = shape->head_dim;
    const int max_splits = int((int64_t(max_ctx) + kSplit - 1) / kSplit);
    Params prm;
    prm.q = static_cast<const __nv_bfloat16*>(q);
    prm.block_table = block_table;
    prm.cu = cu_seqlens_q;
    prm.ctx = ctx_lens;
    prm.items = items;
    prm.ws_acc = static_cast<float*>(workspace);
    prm.ws_ml = workspace ? static_cast<float*>(workspace) +
                                size_t(T) * max_splits * shape->num_q_heads * D
                          : nullptr;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.err = err_flag;
    prm.B = B;
    prm.T = T;
    prm.max_blocks = max_blocks;
    prm.max_splits = max_splits;
    prm.Hq = shape->num_q_heads;
    prm.Hkv = shape->num_kv_heads;
    prm.g = shape->num_q_heads / shape->num_kv_heads;
    prm.bs = shape->block_size;
    prm.num_blocks = shape->num_blocks;
    prm.c = float(1.4426950408889634 / std::sqrt(double(D)));
    if (D == 128) return launch<128>(mk, mv, prm, n_items, B, T, max_ctx, stream);
    return launch<64>(mk, mv, prm, n_items, B, T, max_ctx, stream);
}

// ------------------------------------------- allocation-free variant of the attention step
// Some callers cannot allocate device memory at the point where they run a step: a serving
// process that reserves all GPU memory up front and forbids later cudaMalloc calls, a plug-in
// that only receives tensors from its host framework and has no allocator of its own, or a
// latency-critical loop where cudaMalloc's implicit device synchronisation is not acceptable.
// For them the split-partial scratch lives in the fixed array below instead of a
// caller-provided workspace. Every GPU that loads the library keeps this array until the
// process exits.
namespace {

static __device__ __align__(256) float g_static_scratch[PA_STATIC_SCRATCH_BYTES / sizeof(float)];

constexpr int kMaxDevices = 64;
float* g_static_scratch_addr[kMaxDevices] = {};   // device address per device, set on first use
std::mutex g_static_scratch_mu;

// Host code cannot use g_static_scratch as a pointer (on the host it names a stand-in, not
// device memory): look its device address up once per device, with that device current.
int32_t static_scratch_for_current_device(float** out) {
    int dev = 0;
    int32_t st = note_cuda(cudaGetDevice(&dev));
    if (st) return st;
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    if (!g_static_scratch_addr[dev]) {
        void* ptr = nullptr;
        st = note_cuda(cudaGetSymbolAddress(&ptr, g_static_scratch));
        if (st) return st;
        g_static_scratch_addr[dev] = static_cast<float*>(ptr);
    }
    *out = g_static_scratch_addr[dev];
    return PA_OK;
}

}  // namespace

extern "C" int32_t paged_attention_step_static_scratch(
    const void* q, const void* k_pool, const void* v_pool, const int32_t* block_table,
    int32_t max_blocks, const int32_t* cu_seqlens_q, const int32_t* ctx_lens, int32_t B,
    int32_t T, int32_t max_ctx, const pa_work_item* items, int32_t n_items, void* out,
    const pa_shape* shape, int32_t* err_flag, pa_stream_t stream) {
    int32_t st = check_shape(shape);
    if (st) return st;
    if (B < 0 || T < 0 || n_items < 0 || max_ctx < 0 || max_blocks < 0) return PA_ERR_INVALID;
    if (T == 0 || n_items == 0) return PA_OK;
    if (!q || !k_pool || !v_pool || !block_table || !cu_seqlens_q || !ctx_lens || !items || !out)
        return PA_ERR_INVALID;
    if (int64_t(shape->num_blocks) * shape->block_size > INT32_MAX) return PA_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool) |
         reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15)
        return PA_ERR_INVALID;
    // the partials of this step must fit the fixed array; nothing is launched otherwise
    if (max_ctx > kSplit && pa_workspace_bytes(shape, T, max_ctx) > PA_STATIC_SCRATCH_BYTES)
        return PA_ERR_WORKSPACE;
    float* scratch = nullptr;
    if ((st = static_scratch_for_current_device(&scratch))) return st;

    CUtensorMap mk, mv;
    if ((st = make_pool_map(&mk, k_pool, shape))) return st;
    if ((st = make_pool_map(&mv, v_pool, shape))) return st;
    const int D = shape->head_dim;
    const int max_splits = int((int64_t(max_ctx) + kSplit - 1) / kSplit);
    Params prm;
    prm.q = static_cast<const __nv_bfloat16*>(q);
    prm.block_table = block_table;
    prm.cu = cu_seqlens_q;
    prm.ctx = ctx_lens;
    prm.items = items;
    prm.ws_acc = scratch;
    prm.ws_ml = scratch + size_t(T) * max_splits * shape->num_q_heads * D;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.err = err_flag;
    prm.B = B;
    prm.T = T;
    prm.max_blocks = max_blocks;
    prm.max_splits = max_splits;
    prm.Hq = shape->num_q_heads;
    prm.Hkv = shape->num_kv_heads;
    prm.g = shape->num_q_heads / shape->num_kv_heads;
    prm.bs = shape->block_size;
    prm.num_blocks = shape->num_blocks;
    prm.c = float(1.4426950408889634 / std::sqrt(double(D)));
    if (D == 128) return launch<128>(mk, mv, prm, n_items, B, T, max_ctx, stream);
    return launch<64>(mk, mv, prm, n_items, B, T, max_ctx, stream);
}
