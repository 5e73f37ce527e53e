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
// Work item = (sequence, KV head, tile of up to 128/g query tokens, KV splits): a decode
// row's item reads one split (its splits are folded by the combine kernel), a prefill tile's
// item reads all of its splits and folds them itself in the combine's order. The M = 128
// rows of every MMA are (token, head-in-group) pairs of one KV head, so K/V tiles are shared
// by the g query heads of a group. A decode item simply has one token (g valid rows). Every
// row runs the same instruction sequence whatever the item holds:
//   S  = Q K^T    tcgen05.mma kind::f16, M 128 x N 128 keys x K D, fp32 in TMEM
//   softmax       fp32 online softmax over 128-key tiles aligned to absolute key positions,
//                 with a reference maximum that moves only when the row maximum outgrows it
//                 by 2^8; a row is spread over 4 threads (tcgen05.ld 16x256b); fixed
//                 reduction order
//   O += P V      tcgen05.mma, M 128 x N D x K 128 keys, P rounded to bf16 and written back
//                 into its tile's S buffer in TMEM (A operand from TMEM)
// A tensor-core output element depends only on its own row of A and column of B, so a row's
// bits do not depend on the other rows of the tile; the fixed splits
// [s*PA_SPLIT_TOKENS, (s+1)*PA_SPLIT_TOKENS) and the ascending-order combine make them
// independent of the batch.
//
// Persistent schedule: CTA c (one per SM) walks list c of the plan, which the host deals
// longest item first to the least-loaded list. Warp roles (384 threads): warps 0-7 softmax /
// rescale / epilogue (two warps per TMEM sub-partition, one per 16-lane half), warp 8
// producer (reads the work items, publishes them in a ring, loads each item's Q tile by TMA
// into one of two Q buffers), warp 9 MMA issuer and TMEM owner, warp 10 K loader, warp 11 V
// loader; over an fp8 cache, 512 threads, warps 12-15 expanding the loaded codes to f16. The
// loaders stream tiles by TMA through rings of shared-memory slots across item boundaries; a
// K slot is free again as soon as S has read it, a V slot once PV has. A paged tile is one
// box per block (K: one per 64-column half, V: both halves in one box), issued from all 32
// lanes of the loader warp. TMEM holds two S buffers (S of the next tile is computed while
// the softmax works on the current one; P overwrites the S it came from) and two O
// accumulators used by alternate splits (a split's epilogue or fold overlaps
// the next split's MMAs; the running result of a prefill tile's earlier splits sits in one of
// them). Every wait on an mbarrier is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
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
constexpr int kThreads = 384;
// an fp8 cache adds four warps (12, 14: K; 13, 15: V) that expand the codes the loaders bring
// in, each pair taking half of every tile's rows
template <bool F8>
constexpr int kThreadsFor = F8 ? kThreads + 128 : kThreads;
constexpr uint32_t kTmemCols = 512;     // S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512)
constexpr uint32_t kTmemO = 256;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // one second per wait

static_assert(kSplit % kTileKeys == 0, "splits are whole tiles");
constexpr int kSplitTiles = kSplit / kTileKeys;
static_assert((kSplitTiles & (kSplitTiles - 1)) == 0, "tiles per split: a power of two");
// Growth of a row's maximum (log2 units) tolerated before its softmax reference moves.
constexpr float kLazyLog2 = 8.f;

template <int D>
struct Layout {
    static constexpr int kChunks = D / 64;                  // 128-byte column chunks of a row
    static constexpr int kStagesK = D == 128 ? 2 : 4;       // K ring: a slot frees after S
    static constexpr int kStagesV = D == 128 ? 3 : 6;       // V ring: a slot frees after PV
    static constexpr int kQHalf = kRows * 128;              // one 64-column chunk of a Q tile
    static constexpr int kQBuf = kChunks * kQHalf;
    static constexpr int kKVHalf = kTileKeys * 128;
    static constexpr int kKVTile = kChunks * kKVHalf;       // K (or V) of one key tile
    static constexpr int kQ = 0;                            // two Q buffers
    static constexpr int kK = kQ + 2 * kQBuf;
    static constexpr int kV = kK + kStagesK * kKVTile;
    static constexpr int kBar = kV + kStagesV * kKVTile;    // barriers, item ring, tables
    static constexpr int kBytes = kBar + 1792;
    static constexpr int kAlloc = kBytes + 1024;            // room to align the base to 1024
};

// mbarrier slots (8 bytes each) at Layout::kBar.
// A waiter tests a phase by its parity, which is only sound while the barrier is within one
// phase of the tested one: the previous phase must already be complete and the next one must
// not be able to complete before the test. Barriers that a role waits on only sometimes (or
// that another role can race ahead on) are therefore split by tile or item parity.
enum Bar {
    kKFull = 0,      // + K slot (up to 4): TMA -> MMA (K of the tile landed)
    kVFull = 4,      // + V slot (up to 6): TMA -> softmax (V of the tile landed)
    kQFull = 10,     // + buffer: TMA -> MMA
    kQEmpty = 12,    // + buffer: MMA (after the item's last S) -> producer
    kSFull = 14,     // + K slot of the tile (tile % SK): MMA -> softmax, K loader: S of the
                     //   tile finished, so its K slot is free as well
    kPFull = 18,     // + tile parity: softmax (256 arrivals) -> MMA: P stored, O rescaled, V
                     //   landed and its tail zeroed (the softmax may finish tile t before the
                     //   MMA has seen tile t-1)
    kPVDone = 20,    // + V slot of the tile (tile % SV): MMA -> softmax, MMA, V loader: the PV
                     //   of the tile finished, so its V slot and the S buffer that held its P
                     //   are free (the softmax waits only when it rescales O and at a split's
                     //   end)
    kOFree = 26,     // + buffer: epilogue (256 arrivals) -> MMA
    kDrain = 28,
    kItemFull = 29,  // + slot (4): producer -> everyone: the slot holds the next item
    kItemEmpty = 33, // + slot: consumers (MMA 2, softmax 256, loaders 64 arrivals) -> producer
    // fp8 cache only: the tile's codes have been expanded to f16 in place (K, V: 64 arrivals from
    // the two expander warps; Q: 32 from the producer), which the MMA and softmax wait for
    // instead of the TMA barrier
    kKReady = 37,    // + K slot
    kVReady = 41,    // + V slot
    kQReady = 47,    // + Q buffer
    kNever = 49,     // nothing ever arrives here: the wait-timeout test waits on it
    kSaved = 50,     // softmax (256 arrivals) -> softmax: a GROUP item's rows have saved their
                     //   state, which the RESUME items after it on the list restore
    kNumBars = 51
};
constexpr int kHolderOff = 8 * kNumBars;          // TMEM address written by tcgen05.alloc
constexpr int kAbortOff = kHolderOff + 4;
constexpr int kRingOff = 512;                     // 4 item slots of 64 bytes
constexpr int kTableOff = 768;                    // per loader warp: the item's table entries
constexpr int kTableKeys = 1024;                  // keys whose table entries a loader holds
constexpr int kTableTiles = kTableKeys / kTileKeys;
constexpr int kMaxTableEntries = kTableKeys / 8;  // at the smallest block size, 8 tokens
static_assert(kSplit % kTableKeys == 0, "a split starts a table window");
static_assert(kAbortOff + 4 <= kRingOff, "control area");

struct Params {
    const __nv_bfloat16* k_pool;
    const __nv_bfloat16* v_pool;
    const int32_t* block_table;
    const int32_t* cu;
    const int32_t* ctx;
    const pa_work_item* items;
    float* ws_acc;      // [T][max_splits][Hq][D]
    float* ws_ml;       // [T][max_splits][Hq][2]
    __nv_bfloat16* out;
    int32_t* err;
    int32_t n_items, B, T, max_blocks, max_splits, Hq, Hkv, g, bs, num_blocks;
    float c;            // log2(e) / sqrt(D) (times the K scale of an fp8 cache): softmax
                        // works in base 2 on raw scores
    float v_scale;      // V scale of an fp8 cache (1 for bf16): out = O * (rcp(l) * v_scale)
    unsigned long long never_ns;   // nonzero only in the wait-timeout test: the softmax warps
                                   // first wait this long on kNever, which nothing completes
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

// The MMA warp runs its whole loop with all 32 lanes, so that its control flow never
// diverges; the instructions that one thread must issue take the issuing lane as a predicate.
__device__ __forceinline__ void mbar_arrive_if(uint32_t issue, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t.reg .b64 st;\n\tsetp.ne.b32 q, %1, 0;\n\t"
        "@q mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar), "r"(issue)
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

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void prefetch_l2(const void* a) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

// Warms L2 with the step metadata a CTA reads first, before the grid dependency wait: its first
// work item, and, dealt out over the grid's CTAs and a warp's lanes, the 128-byte lines of
// cu_seqlens_q, ctx_lens and the block table (up to 8 lines a lane). The dependent reads
// after the wait (item, then the sequence's metadata, then its table window) then hit L2. A
// prefetch loads nothing into registers: a preceding kernel's writes to these arrays are still
// what the reads after the wait see.
__device__ __forceinline__ void prefetch_step_meta(const pa_work_item* items, int n_items,
                                                   const int32_t* cu, const int32_t* ctx,
                                                   const int32_t* table, int B, int max_blocks,
                                                   int lane) {
    const int c = int(blockIdx.x);
    if (lane == 0 && items && c < n_items) prefetch_l2(items + c);
    if (!cu || !ctx || !table || B <= 0 || max_blocks <= 0) return;
    const int64_t l_cu = (int64_t(B) + 1 + 31) / 32, l_ctx = (int64_t(B) + 31) / 32;
    const int64_t l_tab = (int64_t(B) * max_blocks + 31) / 32;
    const int64_t total = l_cu + l_ctx + l_tab;
    const int64_t stride = int64_t(gridDim.x) * 32;
    int64_t l = int64_t(c) * 32 + lane;
    for (int k = 0; k < 8 && l < total; ++k, l += stride)
        prefetch_l2(l < l_cu ? cu + l * 32
                    : l < l_cu + l_ctx ? ctx + (l - l_cu) * 32
                                       : table + (l - l_cu - l_ctx) * 32);
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with the given parity. Gives up when another role has set
// the CTA's abort word or after limit_ns; then sets the abort word and returns false.
__device__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_word,
                             unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_word) return false;
        if (global_ns() - t0 > limit_ns) {
            *abort_word = 1;
            return false;
        }
    }
}

// Waits for an mbarrier phase that the CTA's own copies or MMAs complete, before the CTA
// leaves: it ignores the abort word (the copies are in flight whatever happened) but still
// gives up after kWaitLimitNs.
__device__ void wait_drain(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return;
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

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y, int32_t z, int32_t w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit_if(uint32_t issue, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
        "r"(issue)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// The MMA groups of one tile, each in one asm block: the issuing warp shares its scheduler
// with two softmax warps that take most issue slots, so every instruction between two MMAs
// costs tensor-pipe time. The predicates are set once per group, and a step k only adds its
// offset / 16 to the low word of a shared-memory descriptor (the start-address field, bits
// 0-13, never carries: shared addresses stay below 2^18).
//
// S group: D[tmem] = sum_k A_k B_k^T with A = Q, B = K (both K-major in shared memory); step k
// reads 16 columns at byte offset (k / 4) * 16384 + (k % 4) * 32 of both operands.
#define PA_S_STEP(OFF, PRED)                                                                   \
    "add.u32 x, al, " #OFF ";\n\tadd.u32 y, bl, " #OFF ";\n\tmov.b64 a, {x, ah};\n\t"            \
    "mov.b64 b, {y, bh};\n\t@q tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, " PRED ";\n\t"
template <int D>
__device__ __forceinline__ void issue_s_group(uint32_t issue, uint32_t d, uint64_t qdesc,
                                              uint64_t kdesc, uint32_t idesc) {
    static_assert(D == 64 || D == 128, "head_dim");
    if constexpr (D == 128) {
        asm volatile(
            "{\n\t.reg .pred q, pt, pf;\n\t.reg .b32 al, ah, bl, bh, x, y;\n\t.reg .b64 a, b;\n\t"
            "setp.ne.b32 q, %4, 0;\n\tsetp.eq.b32 pt, %4, %4;\n\tsetp.ne.b32 pf, %4, %4;\n\t"
            "mov.b64 {al, ah}, %1;\n\tmov.b64 {bl, bh}, %2;\n\t"
            "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
            PA_S_STEP(2, "pt") PA_S_STEP(4, "pt") PA_S_STEP(6, "pt") PA_S_STEP(1024, "pt")
            PA_S_STEP(1026, "pt") PA_S_STEP(1028, "pt") PA_S_STEP(1030, "pt") "}" ::"r"(d),
            "l"(qdesc), "l"(kdesc), "r"(idesc), "r"(issue)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred q, pt, pf;\n\t.reg .b32 al, ah, bl, bh, x, y;\n\t.reg .b64 a, b;\n\t"
            "setp.ne.b32 q, %4, 0;\n\tsetp.eq.b32 pt, %4, %4;\n\tsetp.ne.b32 pf, %4, %4;\n\t"
            "mov.b64 {al, ah}, %1;\n\tmov.b64 {bl, bh}, %2;\n\t"
            "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
            PA_S_STEP(2, "pt") PA_S_STEP(4, "pt") PA_S_STEP(6, "pt") "}" ::"r"(d), "l"(qdesc),
            "l"(kdesc), "r"(idesc), "r"(issue)
            : "memory");
    }
}
#undef PA_S_STEP

// PV group: D[tmem] (+)= sum_k P_k V_k, P from TMEM (8 packed columns per 16 keys, at p + 8 k),
// V from shared memory (MN-major) at descriptor offset off[k] (off[0] = 0); the first step
// accumulates only when acc is set.
__device__ __forceinline__ void issue_pv_group(uint32_t issue, uint32_t d, uint32_t p_tmem,
                                               uint64_t vdesc, uint32_t idesc, uint32_t acc,
                                               const uint32_t (&off)[8]) {
    asm volatile(
        "{\n\t.reg .pred q, pt, p0;\n\t.reg .b32 vl, vh, x, t;\n\t.reg .b64 b;\n\t"
        "setp.ne.b32 q, %4, 0;\n\tsetp.eq.b32 pt, %4, %4;\n\tsetp.ne.b32 p0, %5, 0;\n\t"
        "mov.b64 {vl, vh}, %2;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p0;\n\t"
        "add.u32 t, %1, 8;\n\tadd.u32 x, vl, %7;\n\tmov.b64 b, {x, vh};\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %3, pt;\n\t"
        "add.u32 t, %1, 16;\n\tadd.u32 x, vl, %8;\n\tmov.b64 b, {x, vh};\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %3, pt;\n\t"
        "add.u32 t, %1, 24;\n\tadd.u32 x, vl, %9;\n\tmov.b64 b, {x, vh};\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %3, pt;\n\t"
        "add.u32 t, %1, 32;\n\tadd.u32 x, vl, %10;\n\tmov.b64 b, {x, vh};\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %3, pt;\n\t"
        "add.u32 t, %1, 40;\n\tadd.u32 x, vl, %11;\n\tmov.b64 b, {x, vh};\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %3, pt;\n\t"
        "add.u32 t, %1, 48;\n\tadd.u32 x, vl, %12;\n\tmov.b64 b, {x, vh};\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %3, pt;\n\t"
        "add.u32 t, %1, 56;\n\tadd.u32 x, vl, %13;\n\tmov.b64 b, {x, vh};\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %3, pt;\n\t"
        "}" ::"r"(d),
        "r"(p_tmem), "l"(vdesc), "r"(idesc), "r"(issue), "r"(acc), "r"(off[0]), "r"(off[1]),
        "r"(off[2]), "r"(off[3]), "r"(off[4]), "r"(off[5]), "r"(off[6]), "r"(off[7])
        : "memory");
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and B bf16 (bits 7-9,
// 10-12 = 1) or both f16 (0), A K-major, B K-major or MN-major (bit 16), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major, bool f16) {
    return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) |
           ((b_mn_major ? 1u : 0u) << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
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

// Packed fp32 pairs (lo, hi) in one 64-bit register for the f32x2 instructions. They are used
// where every row goes through the same instructions whatever its item (the softmax and the
// rescale); the fold of split partials stays scalar like the combine kernel it must match.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Maximum of 32 values (exact in any order).
__device__ __forceinline__ float max32(const float (&v)[32]) {
    float t[11];
#pragma unroll
    for (int k = 0; k < 10; ++k) t[k] = max3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
    t[10] = fmaxf(v[30], v[31]);
    const float u0 = max3(t[0], t[1], t[2]), u1 = max3(t[3], t[4], t[5]);
    const float u2 = max3(t[6], t[7], t[8]), u3 = fmaxf(t[9], t[10]);
    return fmaxf(max3(u0, u1, u2), u3);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Four e4m3 codes (lowest byte first) -> two f16x2 words (exact: every e4m3 value is an f16
// value).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Expands the 128-byte code rows r_begin .. rows - 1 of a K (IS_V false) or V ring slot to f16
// in place (8 lanes per row, 4 rows per pass). rows - r_begin is a multiple of 8 (whole blocks
// of at least 8 rows), so every pass has 4 valid rows. Row R's codes sit unswizzled where the
// row's second 64-column f16 half goes (K slots: [half][key row]; V slots: [block][half][row]);
// its f16 halves go to the 128-byte swizzled rows TMA would have written. A row is read by its
// 8 lanes before any lane writes over it.
template <bool IS_V>
__device__ __forceinline__ void expand_codes(uint32_t slot, int r_begin, int rows, int bs,
                                             int log2bs, int lane) {
    const int c = lane & 7;                    // code chunk: columns 16 c .. 16 c + 15
    const uint32_t j0 = uint32_t(2 * (c & 3)); // its first f16 chunk within the half
    const uint32_t hi = uint32_t(c >> 2);      // the half it goes to
    for (int R0 = r_begin; R0 + 4 <= rows; R0 += 4) {        // warp-uniform: whole passes
        const int R = R0 + (lane >> 3);
        uint32_t b0, half_step;
        if constexpr (IS_V) {
            b0 = slot + uint32_t(R >> log2bs) * uint32_t(bs * 256) + uint32_t(R & (bs - 1)) * 128;
            half_step = uint32_t(bs * 128);
        } else {
            b0 = slot + uint32_t(R) * 128;
            half_step = uint32_t(kTileKeys * 128);
        }
        const uint32_t b1 = b0 + half_step;
        const uint4 v = ld_shared_v4(b1 + uint32_t(c) * 16);
        __syncwarp();
        uint32_t f[8];
        e4m3x4_to_f16x4(v.x, f[0], f[1]);
        e4m3x4_to_f16x4(v.y, f[2], f[3]);
        e4m3x4_to_f16x4(v.z, f[4], f[5]);
        e4m3x4_to_f16x4(v.w, f[6], f[7]);
        const uint32_t rb = b0 + hi * half_step;
        const uint32_t x = uint32_t(R & 7);    // 128-byte swizzle: chunk ^ (row & 7)
        st_shared_v4(rb + ((j0 ^ x) << 4), f[0], f[1], f[2], f[3]);
        st_shared_v4(rb + (((j0 + 1) ^ x) << 4), f[4], f[5], f[6], f[7]);
    }
}

// Two bf16 (lower half first) -> two f16, rounded to nearest and saturated at +-65504.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
        : "=r"(r)
        : "f"(__uint_as_float(w & 0xFFFF0000u)), "f"(__uint_as_float(w << 16)));
    return r;
}
__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
}

// One work item, checked against the metadata it points at (device data). A bad item does
// no work in any role and raises PA_DEVERR_META (reported by the softmax warps).
struct Item {
    bool good;
    int seq, ctx, q_start, n_q, kvh, split, n_splits, pos0, k_begin, n_tiles, rows_valid;
    int kind;           // PA_ITEM_*
    int tile0;          // the item's first key tile within its split: a RESUME item's tile0
                        // (it continues split 0 there), 0 for every other item
};

// What the producer publishes in an item slot (64 bytes); `last` marks the end of the CTA's
// item list.
struct ItemSlot {
    int seq, ctx, q_start, n_q, kvh, split, n_splits, pos0, k_begin, n_tiles, rows_valid, last,
        kind, tile0, pad[2];
};
static_assert(sizeof(ItemSlot) == 64, "item slot size");

__device__ __forceinline__ Item slot_item(const volatile ItemSlot* sl, bool* last) {
    Item I;
    I.good = true;
    I.seq = sl->seq;
    I.ctx = sl->ctx;
    I.q_start = sl->q_start;
    I.n_q = sl->n_q;
    I.kvh = sl->kvh;
    I.split = sl->split;
    I.n_splits = sl->n_splits;
    I.pos0 = sl->pos0;
    I.k_begin = sl->k_begin;
    I.n_tiles = sl->n_tiles;
    I.rows_valid = sl->rows_valid;
    I.kind = sl->kind;
    I.tile0 = sl->tile0;
    *last = sl->last != 0;
    return I;
}

// Called by all 32 lanes of the producer warp (a GROUP item's members are checked one per
// lane).
// A GROUP item covers the decode rows of sequences seq .. seq + n_q - 1 at tokens q_start .. ,
// each with keys past the shared tiles (which are read through seq's table). Lane i checks
// member i; the warp agrees. Out of line, as it runs for GROUP items only.
__device__ __noinline__ bool group_members_ok(const int32_t* cu, const int32_t* ctx, int B,
                                              int bs, int max_blocks, int seq, int n_q,
                                              int q_start, int tile0, int lane) {
    bool good = seq + n_q <= B;
    bool mine = true;
    if (good && lane < n_q) {
        const int s = seq + lane;
        const int c0 = cu[s], c1 = cu[s + 1], cx = ctx[s];
        mine = c1 - c0 == 1 && c0 == q_start + lane && cx > tile0 * kTileKeys &&
               (int64_t(cx) + bs - 1) / bs <= max_blocks;
    }
    return __all_sync(0xffffffffu, good && mine);
}

__device__ __forceinline__ Item load_item(const Params& p, int idx, int lane) {
    const pa_work_item it = p.items[idx];
    Item I;
    const bool shared = it.kind == PA_ITEM_GROUP || it.kind == PA_ITEM_RESUME;
    bool good = it.seq >= 0 && it.seq < p.B && it.kv_head >= 0 && it.kv_head < p.Hkv &&
                it.n_q >= 1 && it.n_q * p.g <= kRows && it.split >= 0 && it.q_start >= 0 &&
                it.q_start + it.n_q <= p.T &&
                (it.kind == PA_ITEM_PLAIN ||
                 (shared && it.split == 0 && it.n_splits <= 1 && it.tile0 >= 1 &&
                  it.tile0 < kSplitTiles && p.ws_acc != nullptr));
    I.kind = good ? it.kind : PA_ITEM_PLAIN;
    I.tile0 = good && it.kind == PA_ITEM_RESUME ? it.tile0 : 0;
    if (good && it.kind == PA_ITEM_GROUP) {
        good = group_members_ok(p.cu, p.ctx, p.B, p.bs, p.max_blocks, it.seq, it.n_q,
                                it.q_start, it.tile0, lane);
        I.good = good;
        I.seq = it.seq;
        I.ctx = it.tile0 * kTileKeys;        // every tile of the item is a whole tile of keys
        I.q_start = it.q_start;
        I.n_q = it.n_q;
        I.kvh = it.kv_head;
        I.split = 0;
        I.n_splits = 1;
        I.pos0 = it.tile0 * kTileKeys - 1;   // no key of the item lies past any row
        I.k_begin = 0;
        I.n_tiles = good ? it.tile0 : 0;
        I.rows_valid = good ? it.n_q * p.g : 0;
        return I;
    }
    const int seq = good ? it.seq : 0;
    const int ctx_s = good ? p.ctx[seq] : 0;
    const int cu0 = good ? p.cu[seq] : 0;
    const int cu1 = good ? p.cu[seq + 1] : 0;
    good = good && cu0 <= it.q_start && it.q_start + it.n_q <= cu1 && cu1 - cu0 <= ctx_s &&
           (int64_t(ctx_s) + p.bs - 1) / p.bs <= p.max_blocks;
    const int pos0 = ctx_s - cu1 + it.q_start;              // position of the item's first row
    const int p_max = pos0 + it.n_q - 1;
    // a RESUME item continues its row's split 0 at key tile tile0
    const int k_begin = I.kind == PA_ITEM_RESUME ? I.tile0 * kTileKeys : it.split * kSplit;
    good = good && k_begin <= p_max && (p_max < kSplit || p_max / kSplit < p.max_splits);
    // a decode row's splits are separate items (folded by the combine kernel); a prefill
    // tile's item starts at split 0 and covers every split its last row reaches
    const int ns = max(it.n_splits, 1);
    good = good && (cu1 - cu0 == 1 ? ns == 1 : it.split == 0 && ns == p_max / kSplit + 1) &&
           (I.kind != PA_ITEM_RESUME || cu1 - cu0 == 1);
    const int k_end = min(it.split * kSplit + ns * kSplit, p_max + 1);
    I.good = good;
    I.seq = seq;
    I.ctx = ctx_s;
    I.q_start = it.q_start;
    I.n_q = it.n_q;
    I.kvh = it.kv_head;
    I.split = it.split;
    I.n_splits = ns;
    I.pos0 = pos0;
    I.k_begin = k_begin;
    I.n_tiles = good ? (k_end - k_begin + kTileKeys - 1) / kTileKeys : 0;
    I.rows_valid = good ? it.n_q * p.g : 0;
    return I;
}

// ---------------------------------------------------------------- the per-row routine
// Every query row, whichever kernel runs it, goes through these three functions, so that its
// bits depend only on its own scores. A thread owns two rows of a 16-row half of the 128-row
// tile (rows r0 + rs and r0 + rs + 8, rs = lane / 4), each spread over the 4 threads
// q4 = lane % 4 (tcgen05.ld 16x256b layout: columns 8 cc + 2 q4 + {0, 1}).
struct Rows2 {
    int pos[2];        // absolute position of the row, -1 for a padding row
    float m[2], l[2];  // softmax reference maximum (raw score units) and running sum
};

__device__ __forceinline__ void rows_init(Rows2& R, int r0, int rs, int rows_valid, int pos0,
                                          int g) {
#pragma unroll
    for (int sr = 0; sr < 2; ++sr) {
        const int row = r0 + rs + 8 * sr;
        R.pos[sr] = row < rows_valid ? pos0 + row / g : -1;
        R.m[sr] = -INFINITY;
        R.l[sr] = 0.f;
    }
}

// Online softmax step of one 128-key tile (keys kb .. kb + 127) for the thread's first NR rows
// (sr = 0 .. NR-1), taken in lockstep so that the two rows' dependency chains interleave: the
// rows' state is updated, their P, rounded to bf16, goes to pk (packed column 4 cc + q4 of row
// sr is pk[2 cc + sr]) and alpha[sr] is the factor the row's O must be scaled by. The
// arithmetic of a row depends on its own scores only.
template <int NR, bool H16>
__device__ __forceinline__ void softmax_rows(const uint32_t (&r)[64], uint32_t (&pk)[32], int q4,
                                             int kb, float c, Rows2& R, float alpha[2]) {
    float sv[NR][32];
    float mx[NR];
#pragma unroll
    for (int sr = 0; sr < NR; ++sr) {
        const int pr = R.pos[sr];
        // the causal / ctx mask matters only when some key of the tile lies past some row of
        // this 8-row block
        if (__all_sync(0xffffffffu, kb + kTileKeys - 1 <= pr)) {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    sv[sr][2 * cc + e] = __uint_as_float(r[4 * cc + 2 * sr + e]);
        } else {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = kb + 8 * cc + 2 * q4 + e;
                    sv[sr][2 * cc + e] =
                        key <= pr ? __uint_as_float(r[4 * cc + 2 * sr + e]) : -INFINITY;
                }
        }
        mx[sr] = max32(sv[sr]);
    }
#pragma unroll
    for (int sr = 0; sr < NR; ++sr) mx[sr] = fmaxf(mx[sr], __shfl_xor_sync(0xffffffffu, mx[sr], 1));
#pragma unroll
    for (int sr = 0; sr < NR; ++sr) mx[sr] = fmaxf(mx[sr], __shfl_xor_sync(0xffffffffu, mx[sr], 2));
    float a[NR], m_ref[NR];
    uint64_t nmc2[NR];
#pragma unroll
    for (int sr = 0; sr < NR; ++sr) {
        // The reference maximum moves only when the row's maximum grows past it by more than
        // 8 in base-2 units, so P <= 2^8 and O needs rescaling rarely; the decision depends on
        // the row's own scores alone.
        const float m_old = R.m[sr];
        const float m_new = fmaxf(m_old, mx[sr]);
        const bool move = m_old == -INFINITY ? m_new != -INFINITY
                                             : __fmul_rn(__fsub_rn(m_new, m_old), c) > kLazyLog2;
        m_ref[sr] = move ? m_new : m_old;
        const float m_use = m_ref[sr] == -INFINITY ? 0.f : m_ref[sr];
        // A row that has not seen a key yet (a padding row of the block, or a row whose
        // position precedes this split) has O = 0 and l = 0: its factor stays 1 so that it
        // never asks for a rescale of O.
        a[sr] = (m_old == m_use || m_ref[sr] == -INFINITY)
                    ? 1.f
                    : ex2(__fmul_rn(__fsub_rn(m_old, m_use), c));
        const float nmc = __fmul_rn(-m_use, c);
        nmc2[sr] = f2(nmc, nmc);
    }
    // p = 2^(s c - m c) for the thread's 32 keys of each row (pairs of adjacent columns
    // packed), then their sum as a fixed tree: the pairs' lanes are added level by level and
    // the two lanes last
    const uint64_t c2 = f2(c, c);
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int sr = 0; sr < NR; ++sr) {
            float x0, x1;
            f2_split(fma2(f2(sv[sr][2 * i], sv[sr][2 * i + 1]), c2, nmc2[sr]), x0, x1);
            sv[sr][2 * i] = ex2(x0);
            sv[sr][2 * i + 1] = ex2(x1);
        }
    uint64_t t8[NR][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int sr = 0; sr < NR; ++sr)
            t8[sr][i] = add2(f2(sv[sr][4 * i], sv[sr][4 * i + 1]),
                             f2(sv[sr][4 * i + 2], sv[sr][4 * i + 3]));
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i)
#pragma unroll
            for (int sr = 0; sr < NR; ++sr) t8[sr][i] = add2(t8[sr][i], t8[sr][i + w]);
    float sum[NR];
#pragma unroll
    for (int sr = 0; sr < NR; ++sr) {
        float lo, hi;
        f2_split(t8[sr][0], lo, hi);
        sum[sr] = __fadd_rn(lo, hi);
    }
#pragma unroll
    for (int sr = 0; sr < NR; ++sr)
        sum[sr] = __fadd_rn(sum[sr], __shfl_xor_sync(0xffffffffu, sum[sr], 1));
#pragma unroll
    for (int sr = 0; sr < NR; ++sr)
        sum[sr] = __fadd_rn(sum[sr], __shfl_xor_sync(0xffffffffu, sum[sr], 2));
#pragma unroll
    for (int sr = 0; sr < NR; ++sr) {
        R.l[sr] = __fadd_rn(__fmul_rn(R.l[sr], a[sr]), sum[sr]);
        R.m[sr] = m_ref[sr];
        alpha[sr] = a[sr];
    }
    // keys 8cc + 2q4 + {0, 1} -> packed column 4cc + q4 (16x128b layout)
#pragma unroll
    for (int cc = 0; cc < 16; ++cc)
#pragma unroll
        for (int sr = 0; sr < NR; ++sr)
            pk[2 * cc + sr] = H16 ? pack_f16(sv[sr][2 * cc], sv[sr][2 * cc + 1])
                                  : pack_bf16(sv[sr][2 * cc], sv[sr][2 * cc + 1]);
}

// Online softmax of one 128-key tile for the half at TMEM address tm_s (lane offset
// included): S is read, the rows' state is updated and P, rounded to bf16, is stored over the
// first 64 columns (as f16 when H16, the operand type of an fp8 cache's MMAs, else bf16).
// alpha[sr] is the factor the row's O must be scaled by. A second 8-row block with no valid
// row (the tail of a decode or of a ragged tile) needs no softmax: its P is never used for a
// written output.
template <bool H16>
__device__ __forceinline__ void softmax_half(uint32_t tm_s, int r0, int q4, int rows_valid,
                                             int kb, float c, Rows2& R, float alpha[2]) {
    uint32_t r[64];
    tmem_ld_16x256b_x16(tm_s, r);
    tmem_wait_ld();
    uint32_t pk[32];                 // P rounded to bf16, packed in pairs
    if (r0 + 8 >= rows_valid) {
        softmax_rows<1, H16>(r, pk, q4, kb, c, R, alpha);
        alpha[1] = 1.f;
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) pk[2 * cc + 1] = 0u;
    } else {
        softmax_rows<2, H16>(r, pk, q4, kb, c, R, alpha);
    }
    // P replaces S in the first 64 columns of this tile's S buffer
    tmem_st_16x128b_x16(tm_s, pk);
}

// O of the half (TMEM address tm_o, lane offset included) scaled row by row by alpha.
template <int D>
__device__ __forceinline__ void rescale_half(uint32_t tm_o, const float alpha[2]) {
    uint32_t o[D / 2];
    if constexpr (D == 128) tmem_ld_16x256b_x16(tm_o, o);
    else tmem_ld_16x256b_x8(tm_o, o);
    tmem_wait_ld();
    const uint64_t a2[2] = {f2(alpha[0], alpha[0]), f2(alpha[1], alpha[1])};
#pragma unroll
    for (int cc = 0; cc < D / 8; ++cc)
#pragma unroll
        for (int sr = 0; sr < 2; ++sr) {
            const int k = 4 * cc + 2 * sr;
            float x0, x1;
            f2_split(mul2(f2(__uint_as_float(o[k]), __uint_as_float(o[k + 1])), a2[sr]), x0, x1);
            o[k] = __float_as_uint(x0);
            o[k + 1] = __float_as_uint(x1);
        }
    if constexpr (D == 128) tmem_st_16x256b_x16(tm_o, o);
    else tmem_st_16x256b_x8(tm_o, o);
}

// Epilogue of the half, O already in registers: a row whose position lies in one split is
// finished here (out = bf16(O * (rcp(l) * v_scale))); a row spanning several splits stores this split's
// partial (acc = O, m, l) for the fixed-order combine. Rows are those of a tile whose first
// row is token q_start at position pos0 (rows_valid rows, g heads per token).
// A GROUP item (save) stores every valid row as the partial of split 0, whatever the row's
// own position: the state its RESUME item restores and continues.
template <int D>
__device__ __forceinline__ void store_half(const Params& p, const uint32_t* o, int r0, int rs,
                                           int q4, int rows_valid, int q_start, int kvh,
                                           int split, const Rows2& R, bool save) {
#pragma unroll
    for (int sr = 0; sr < 2; ++sr) {
        const int row = r0 + rs + 8 * sr;
        if (row >= rows_valid) continue;
        const int pr = R.pos[sr];
        const int nsp = pr / kSplit + 1;
        if (split >= nsp) continue;              // the row has no keys in this split
        const int tok = q_start + row / p.g;
        const int head = kvh * p.g + row % p.g;
        if (nsp == 1 && !save) {
            const float inv = __fmul_rn(__frcp_rn(R.l[sr]), p.v_scale);
            __nv_bfloat16* dst = p.out + (int64_t(tok) * p.Hq + head) * D;
#pragma unroll
            for (int cc = 0; cc < D / 8; ++cc) {
                const float x0 = __fmul_rn(__uint_as_float(o[4 * cc + 2 * sr]), inv);
                const float x1 = __fmul_rn(__uint_as_float(o[4 * cc + 2 * sr + 1]), inv);
                *reinterpret_cast<uint32_t*>(dst + 8 * cc + 2 * q4) = pack_bf16(x0, x1);
            }
        } else {
            const int64_t slot = (int64_t(tok) * p.max_splits + split) * p.Hq + head;
            float* acc = p.ws_acc + slot * D;
#pragma unroll
            for (int cc = 0; cc < D / 8; ++cc)
                *reinterpret_cast<float2*>(acc + 8 * cc + 2 * q4) =
                    make_float2(__uint_as_float(o[4 * cc + 2 * sr]),
                                __uint_as_float(o[4 * cc + 2 * sr + 1]));
            if (q4 == 0)
                *reinterpret_cast<float2*>(p.ws_ml + slot * 2) = make_float2(R.m[sr], R.l[sr]);
        }
    }
}

// Start of a RESUME item: the rows' state saved by their GROUP item is restored, (m, l) into the
// returned rows and the accumulator into the item's O buffer (TMEM address tm_o, lane offset
// included), so that the row continues its split exactly where it would have been without the
// sharing. Out of line: it runs once per RESUME item, and inlined it would sit in the body of
// the persistent loop that every other item runs.
template <int D>
__device__ __noinline__ Rows2 restore_half(const float* ws_acc, const float* ws_ml, int g,
                                           int max_splits, int Hq, uint32_t tm_o, int r0, int rs,
                                           int q4, int rows_valid, int q_start, int kvh,
                                           int pos0) {
    Rows2 R;
    uint32_t o[D / 2];
#pragma unroll
    for (int sr = 0; sr < 2; ++sr) {
        const int row = r0 + rs + 8 * sr;
        const bool valid = row < rows_valid;
        R.pos[sr] = valid ? pos0 + row / g : -1;
        R.m[sr] = -INFINITY;
        R.l[sr] = 0.f;
        const int64_t slot = valid ? int64_t(q_start + row / g) * max_splits * Hq + kvh * g +
                                         row % g
                                   : 0;
        if (valid) {
            const float2 ml = *reinterpret_cast<const float2*>(ws_ml + slot * 2);
            R.m[sr] = ml.x;
            R.l[sr] = ml.y;
        }
        const float* acc = ws_acc + slot * D;
#pragma unroll
        for (int cc = 0; cc < D / 8; ++cc) {
            const float2 v = valid ? *reinterpret_cast<const float2*>(acc + 8 * cc + 2 * q4)
                                   : make_float2(0.f, 0.f);
            o[4 * cc + 2 * sr] = __float_as_uint(v.x);
            o[4 * cc + 2 * sr + 1] = __float_as_uint(v.y);
        }
    }
    if constexpr (D == 128) tmem_st_16x256b_x16(tm_o, o);
    else tmem_st_16x256b_x8(tm_o, o);
    tmem_wait_st();
    return R;
}

// Running result of a prefill tile's splits 0 .. j-1, per row: reference maximum and sum
// (its accumulator stays in TMEM).
struct Fold2 {
    float M[2], L[2];
};

// End of split js >= 1 of an item that covers all splits of its rows: the split's partial (O
// at TMEM address tm_p, the rows' (m, l) in R) is folded into the running result of the
// earlier splits (accumulator at tm_a, (M, L) in F) with the split combine's arithmetic, in
// the same order: M' = max(M, m), a = 2^((M - M') c), b = 2^((m - M') c), L = L a + l b,
// ACC = ACC a + O b. A row whose position precedes the split has no keys in it and keeps its
// running result unchanged, as the combine would not fold it. Unless fin, the result goes to
// tm_p, whose buffer holds the running result from here on; with fin the rows are finished,
// out = bf16(ACC * (rcp(L) * v_scale)), like every other row of the step.
template <int D>
__device__ __forceinline__ void fold_half(const Params& p, uint32_t tm_a, uint32_t tm_p, int r0,
                                          int rs, int q4, int rows_valid, int q_start, int kvh,
                                          int js, bool fin, const Rows2& R, Fold2& F) {
    float fa[2], fb[2], inv[2];
    bool take[2];
#pragma unroll
    for (int sr = 0; sr < 2; ++sr) {
        take[sr] = R.pos[sr] >= js * kSplit;
        fa[sr] = 1.f;
        fb[sr] = 0.f;
        if (take[sr]) {
            const float mn = fmaxf(F.M[sr], R.m[sr]);
            fa[sr] = F.M[sr] == mn ? 1.f : ex2(__fmul_rn(__fsub_rn(F.M[sr], mn), p.c));
            fb[sr] = R.m[sr] == mn ? 1.f : ex2(__fmul_rn(__fsub_rn(R.m[sr], mn), p.c));
            F.L[sr] = __fadd_rn(__fmul_rn(F.L[sr], fa[sr]), __fmul_rn(R.l[sr], fb[sr]));
            F.M[sr] = mn;
        }
        inv[sr] = fin ? __fmul_rn(__frcp_rn(F.L[sr]), p.v_scale) : 0.f;
    }
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
        uint32_t a[32], o[32];
        tmem_ld_16x256b_x8(tm_a + 64 * h, a);
        tmem_ld_16x256b_x8(tm_p + 64 * h, o);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
#pragma unroll
            for (int sr = 0; sr < 2; ++sr) {
                if (!take[sr]) continue;
                // scalar, like the combine kernel: packed multiplies feeding a packed add
                // may be contracted into a fused multiply-add, which rounds once and can
                // differ from the combine's result in the last bit
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = 4 * cc + 2 * sr + e;
                    a[k] = __float_as_uint(__fadd_rn(__fmul_rn(__uint_as_float(a[k]), fa[sr]),
                                                     __fmul_rn(__uint_as_float(o[k]), fb[sr])));
                }
            }
        if (!fin) {
            tmem_st_16x256b_x8(tm_p + 64 * h, a);
            continue;
        }
#pragma unroll
        for (int sr = 0; sr < 2; ++sr) {
            const int row = r0 + rs + 8 * sr;
            if (row >= rows_valid) continue;
            const int tok = q_start + row / p.g;
            const int head = kvh * p.g + row % p.g;
            __nv_bfloat16* dst = p.out + (int64_t(tok) * p.Hq + head) * D + 64 * h;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const float x0 = __fmul_rn(__uint_as_float(a[4 * cc + 2 * sr]), inv[sr]);
                const float x1 = __fmul_rn(__uint_as_float(a[4 * cc + 2 * sr + 1]), inv[sr]);
                *reinterpret_cast<uint32_t*>(dst + 8 * cc + 2 * q4) = pack_bf16(x0, x1);
            }
        }
    }
    if (!fin) tmem_wait_st();
}

// Keys at or beyond ctx in the tile starting at key kb are stale or were never loaded: their
// V rows in the slot at vb are zeroed (threads tid of nthr share the work) so that their zero
// probabilities contribute exact zeros.
template <int D>
__device__ __forceinline__ void zero_v_tail(uint32_t vb, int kb, int ctx, int bs, int tid,
                                            int nthr) {
    constexpr int kChunks = D / 64;
    const int z0 = max(ctx - kb, 0);
    const int nrow = kTileKeys - z0;
    for (int i = tid; i < nrow * 8 * kChunks; i += nthr) {
        const int hh = i / (nrow * 8);
        const int rem = i % (nrow * 8);
        const int key = z0 + rem / 8;
        st_shared_zero16(vb + (key / bs) * (bs * 128 * kChunks) + hh * (bs * 128) +
                         (key % bs) * 128 + (rem % 8) * 16);
    }
}

// F8: the pools hold float8_e4m3fn codes (head_dim 128 only); the loaders expand each tile
// to f16 in shared memory, Q is rounded to f16, and the MMAs take f16 operands.
template <int D, bool F8>
__global__ void __launch_bounds__(kThreadsFor<F8>, 1)
    paged_attn_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q1,
                      const __grid_constant__ CUtensorMap tm_qn, const Params p) {
    using L = Layout<D>;
    static_assert(!F8 || D == 128, "the fp8 cache is supported at head_dim 128");
    constexpr int SK = L::kStagesK;
    static_assert(SK == 2 || SK == 4, "K ring slots: 2 or 4");
    constexpr int kLog2SK = SK == 2 ? 1 : 2;
    // what the MMA and softmax wait for: the TMA landing, or (fp8 cache) the f16 expansion
    constexpr int kKUse = F8 ? kKReady : kKFull;
    constexpr int kVUse = F8 ? kVReady : kVFull;
    constexpr int kQUse = F8 ? kQReady : kQFull;
    constexpr int SV = L::kStagesV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t bars = sb + L::kBar;
    volatile int* abort_word = reinterpret_cast<volatile int*>(smem + L::kBar + kAbortOff);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const auto bar = [&](int b) { return bars + 8 * b; };

    if (warp == 8)
        prefetch_step_meta(p.items, p.n_items, p.cu, p.ctx, p.block_table, p.B, p.max_blocks,
                           lane);
    if (threadIdx.x == 0) {
        for (int b = 0; b < kNumBars; ++b)
            mbar_init(bars + 8 * b,
                      (b == kPFull || b == kPFull + 1 || b == kOFree || b == kOFree + 1 ||
                       b == kSaved) ? 256
                      : (b >= kItemEmpty && b < kItemEmpty + 4)       ? 2 + 256 + 64 + (F8 ? 128 : 0)
                      : (b >= kKReady && b < kQReady)                 ? 64
                      : b >= kQReady                                  ? 32
                                                                      : 1);
        *abort_word = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 9) {
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
    // launched as a programmatic dependent: nothing written by the previous kernel on the
    // stream (the KV write, or whatever produced q) is read before this point
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        // Reads the work items from global memory, publishes each one in a slot of the item
        // ring for the other roles, and loads its Q tile by TMA.
        volatile ItemSlot* ring = reinterpret_cast<volatile ItemSlot*>(smem + L::kBar + kRingOff);
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q1)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_qn)) : "memory");
        }
        int ic = 0;
        int ok = 1;
        // The plan's list blockIdx.x: it starts at that item and follows `next`, which only
        // moves forward, so the walk ends. Padding (n_q == 0) ends it too.
        int idx = int(blockIdx.x);
        for (;;) {
            Item I;
            I.good = false;
            bool have = false;
            while (idx >= 0 && idx < p.n_items) {
                const int cur = idx;
                // an item with n_q == 0 is padding (a plan padded to a fixed item count, so
                // that a captured step can be replayed with new metadata): no more work
                if (p.items[cur].n_q == 0) break;
                const int nxt = p.items[cur].next;
                if (nxt > 0 && (nxt <= cur || nxt >= p.n_items)) {
                    if (lane == 0 && p.err) atomicOr(p.err, PA_DEVERR_META);
                    idx = -1;                             // a link that does not move forward
                } else {
                    idx = nxt > 0 ? nxt : -1;
                }
                I = load_item(p, cur, lane);
                if (I.good) {
                    have = true;
                    break;
                }
                if (lane == 0 && p.err) atomicOr(p.err, PA_DEVERR_META);
            }
            // out of items: the dependent combine may start launching as CTAs retire
            if (!have && lane == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            const int slot = ic & 3;
            if (lane == 0) {
                if (ic >= 4)
                    ok = wait_bounded(bar(kItemEmpty + slot), ((ic >> 2) - 1) & 1, abort_word);
                if (ok) {
                    volatile ItemSlot* sl = ring + slot;
                    sl->seq = I.seq;
                    sl->ctx = I.ctx;
                    sl->q_start = I.q_start;
                    sl->n_q = I.n_q;
                    sl->kvh = I.kvh;
                    sl->split = I.split;
                    sl->n_splits = I.n_splits;
                    sl->pos0 = I.pos0;
                    sl->k_begin = I.k_begin;
                    sl->n_tiles = I.n_tiles;
                    sl->rows_valid = I.rows_valid;
                    sl->kind = I.kind;
                    sl->tile0 = I.tile0;
                    sl->last = have ? 0 : 1;
                    mbar_arrive(bar(kItemFull + slot));
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok || !have) break;
            // Q: rows (token, head-in-group), one box per 64-column chunk
            const int qb = ic & 1;
            if (lane == 0 && ic >= 2)
                ok = wait_bounded(bar(kQEmpty + qb), ((ic >> 1) - 1) & 1, abort_word);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                const bool dec = I.n_q == 1;
                const CUtensorMap* tq = dec ? &tm_q1 : &tm_qn;
                const uint32_t rows = dec ? uint32_t(p.g) : uint32_t(kRows);
                mbar_expect_tx(bar(kQFull + qb), rows * 128 * L::kChunks);
                for (int h = 0; h < L::kChunks; ++h)
                    tma_load_3d(sb + L::kQ + qb * L::kQBuf + h * L::kQHalf, tq, bar(kQFull + qb),
                                64 * h, I.kvh * p.g, I.q_start);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if constexpr (F8) {
                // the MMAs of an fp8 cache take f16 operands: once Q has landed, round it to
                // f16 in place (every 16-byte chunk keeps its position, so the swizzle holds)
                if (lane == 0) ok = wait_bounded(bar(kQFull + qb), (ic >> 1) & 1, abort_word);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const int rows = I.n_q == 1 ? p.g : kRows;
                const uint32_t qbase = sb + L::kQ + qb * L::kQBuf;
                for (int i = lane; i < rows * 8 * L::kChunks; i += 32) {
                    const int r = i / (8 * L::kChunks);
                    const int rem = i - r * 8 * L::kChunks;
                    const uint32_t a = qbase + (rem >> 3) * L::kQHalf + r * 128 + (rem & 7) * 16;
                    const uint4 v = ld_shared_v4(a);
                    st_shared_v4(a, bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y),
                                 bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
                }
                fence_proxy_async();
                __syncwarp();
                mbar_arrive(bar(kQReady + qb));          // all 32 lanes arrive
            }
            ++ic;
        }
        if (lane == 0) {
            // never leave with copies in flight into this CTA's shared memory
            for (int i = max(0, ic - 2); i < ic; ++i)
                wait_drain(bar(kQFull + (i & 1)), (i >> 1) & 1);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        // Lane 0 alone runs the loop: the warp shares its scheduler with two softmax warps,
        // and every instruction it issues between MMA groups leaves the tensor pipe idle, so
        // no warp-wide work is spent on it (the other lanes wait at the final barrier).
        if (lane == 0) {
            const uint32_t leader = 1u;
            constexpr uint32_t idesc_s = make_idesc(kRows, kTileKeys, false, F8);
            constexpr uint32_t idesc_o = make_idesc(kRows, D, true, F8);
            static_assert(L::kQHalf == L::kKVHalf, "Q and K chunks share the step offsets");
            // This warp shares its scheduler with two softmax warps, and tcgen05.mma issue
            // takes about as long as the tensor work, so every instruction of this loop costs
            // tensor-pipe time: descriptors are built once per buffer, and a 16-wide step k
            // only adds its byte offset / 16 to the start-address field (bits 0-13; shared
            // addresses stay below 2^18, so the add never carries out of the field).
            const uint64_t qd0 = make_sdesc(sb + L::kQ, 16, 1024);
            const uint64_t kd0 = make_sdesc(sb + L::kK, 16, 1024);
            constexpr uint32_t kBufStep = uint32_t(L::kKVTile) >> 4;
            static_assert(L::kQBuf == L::kKVTile, "Q buffers and K/V slots have one size");
            static_assert(L::kQHalf == 16384, "the S group's step offsets");
            const auto issue_s = [&](uint64_t qdesc, uint64_t kdesc, uint32_t d) {
                issue_s_group<D>(leader, d, qdesc, kdesc, idesc_s);
            };
            // V tile: block b of the tile at b * bs * 128 * chunks bytes, its 64-column halves
            // bs * 128 bytes apart (MN-major B operand: LBO = half stride, SBO = 8-key stride)
            const uint32_t v_lbo = uint32_t(p.bs) * 128;
            const uint32_t v_sbo = p.bs >= 16 ? 1024u : uint32_t(p.bs) * 128 * L::kChunks;
            const uint64_t vd0 = make_sdesc(sb + L::kV, v_lbo, v_sbo);
            // offset / 16 of the 16-key step k inside a V slot (block of the step, row in the
            // block), computed once
            uint32_t v_off[kTileKeys / 16];
            {
                const int log2bs = __ffs(p.bs) - 1;
#pragma unroll
                for (int k = 0; k < kTileKeys / 16; ++k) {
                    const int key = 16 * k;
                    v_off[k] = (uint32_t(key >> log2bs) * (uint32_t(p.bs) * 128 * L::kChunks) +
                                uint32_t(key & (p.bs - 1)) * 128) >> 4;
                }
            }
            static_assert(kTileKeys / 16 == 8, "eight PV steps per tile");
            const auto issue_pv = [&](uint64_t vdesc, uint32_t p_tmem, uint32_t d, bool acc) {
                // P of keys 16k .. 16k+15 is 8 packed columns of the S buffer
                issue_pv_group(leader, d, p_tmem, vdesc, idesc_o, acc ? 1u : 0u, v_off);
            };
            // Two cursors walk the same item sequence: one issues S = Q K^T for the next tile
            // as soon as its K has landed (and its S buffer is free), the other issues O += P V
            // as soon as the softmax has produced P. Neither waits for the other, so the
            // stage of a finished tile is released without waiting for the next tile's data.
            // Each split of an item (its tiles from a multiple of kSplitTiles on) accumulates
            // in an O buffer of its own, alternating with the split counter sg. vs / vph follow
            // tc % SV and (tc / SV) & 1 (the V ring's slot and phase).
            struct Cursor {
                int ic, jt, tc, sg, vs, vph;
                bool have, done;
                Item I;
            };
            const volatile ItemSlot* ring =
                reinterpret_cast<const volatile ItemSlot*>(smem + L::kBar + kRingOff);
            // takes the cursor's next item from the ring once the producer has published it
            const auto fetch = [&](Cursor& c) {
                if (c.have || c.done) return;
                const int slot = c.ic & 3;
                if (!mbar_test_wait(bar(kItemFull + slot), (c.ic >> 2) & 1)) return;
                bool last;
                c.I = slot_item(ring + slot, &last);
                mbar_arrive_if(leader, bar(kItemEmpty + slot));
                c.have = !last;
                c.done = last;
            };
            const auto advance = [&](Cursor& c) {
                ++c.tc;
                if (++c.vs == SV) {
                    c.vs = 0;
                    c.vph ^= 1;
                }
                if (++c.jt == c.I.n_tiles) {
                    c.jt = 0;
                    ++c.ic;
                    ++c.sg;
                    c.have = false;
                } else if ((c.jt & (kSplitTiles - 1)) == 0) {
                    ++c.sg;
                }
            };
            Cursor cs{0, 0, 0, 0, 0, 0, false, false, Item{}};
            Cursor cv{0, 0, 0, 0, 0, 0, false, false, Item{}};
            unsigned idle = 0;
            unsigned long long idle_since = 0;
            while (!(cs.done && cv.done)) {
                bool progress = false;
                fetch(cv);
                fetch(cs);
                // O += P V for the oldest tile whose P is ready (P published implies that V
                // has landed; the first tile of a split starts its O buffer once the epilogue
                // has released it)
                // (a RESUME item's first tile continues its split: it accumulates onto the
                // restored O)
                const bool cont = ((cv.I.tile0 + cv.jt) & (kSplitTiles - 1)) != 0;
                if (cv.have && cv.tc < cs.tc &&
                    mbar_test_wait(bar(kPFull + (cv.tc & 1)), (cv.tc >> 1) & 1) &&
                    (cont || cv.sg < 2 ||
                     mbar_test_wait(bar(kOFree + (cv.sg & 1)), ((cv.sg >> 1) - 1) & 1))) {
                    tc_fence_after();
                    issue_pv(vd0 + uint32_t(cv.vs) * kBufStep, tmem + (cv.tc & 1) * 128,
                             tmem + kTmemO + (cv.sg & 1) * 128, cont);
                    tc_commit_if(leader, bar(kPVDone + cv.vs));
                    advance(cv);
                    progress = true;
                }
                // S = Q K^T for the next tile: its S buffer last held the P of tile cs.tc - 2,
                // which must have been read by that tile's PV (finished, not just issued);
                // that PV's barrier is V slot (tc - 2) % SV, phase ((tc - 2) / SV) & 1
                const int ks = cs.tc & (SK - 1);
                const int pv2 = cs.vs >= 2 ? cs.vs - 2 : cs.vs - 2 + SV;
                const int pv2ph = cs.vs >= 2 ? cs.vph : cs.vph ^ 1;
                if (cs.have && cs.tc <= cv.tc + 1 &&
                    (cs.tc < 2 || mbar_test_wait(bar(kPVDone + pv2), pv2ph)) &&
                    (cs.jt > 0 || mbar_test_wait(bar(kQUse + (cs.ic & 1)), (cs.ic >> 1) & 1)) &&
                    mbar_test_wait(bar(kKUse + ks), (cs.tc >> kLog2SK) & 1)) {
                    tc_fence_after();
                    issue_s(qd0 + uint32_t(cs.ic & 1) * kBufStep, kd0 + uint32_t(ks) * kBufStep,
                            tmem + (cs.tc & 1) * 128);
                    tc_commit_if(leader, bar(kSFull + ks));
                    tc_commit_if(leader && cs.jt == cs.I.n_tiles - 1, bar(kQEmpty + (cs.ic & 1)));
                    advance(cs);
                    progress = true;
                }
                // the clock is read every 64 idle polls only
                if (progress) {
                    idle = 0;
                } else if ((++idle & 63) == 0) {
                    if (*abort_word) break;
                    const unsigned long long now = global_ns();
                    if (idle == 64) {
                        idle_since = now;
                    } else if (now - idle_since > kWaitLimitNs) {
                        *abort_word = 1;
                        break;
                    }
                }
            }
            // drain: every MMA lane 0 issued has finished before TMEM is released
            tc_commit_if(leader, bar(kDrain));
            wait_drain(bar(kDrain), 0);
        }
    } else if (warp == 10 || warp == 11) {
        // ------------------------------------------------------------ K (warp 10) / V (warp 11)
        const bool is_v = warp == 11;
        int32_t* tbl = reinterpret_cast<int32_t*>(smem + L::kBar + kTableOff) +
                       (warp - 10) * kMaxTableEntries;
        const volatile ItemSlot* ring =
            reinterpret_cast<const volatile ItemSlot*>(smem + L::kBar + kRingOff);
        const CUtensorMap* tmap = is_v ? &tm_v : &tm_k;
        if (lane == 0)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
        const int log2bs = __ffs(p.bs) - 1;
        // boxes per block: K one per 64-column half; V one (both halves) when D = 128
        const int boxes_per_block = is_v ? 1 : L::kChunks;
        const int full_b = is_v ? kVFull : kKFull;
        // a K slot is free once S of its tile has finished, a V slot once PV has
        const int empty_b = is_v ? kPVDone : kSFull;
        const int S = is_v ? SV : SK;                    // slots in this tensor's ring
        const uint32_t slots = sb + (is_v ? L::kV : L::kK);
        int tc = 0, ic = 0;
        int ok = 1;
        // fp8 cache: shared address of row R of a slot's 64-column half h (K: [half][key row];
        // V: [block][half][row]). The codes of row R land unswizzled at row_base(R, 1), where
        // the row's second f16 half goes, and are expanded there (expand_codes).
        const auto row_base = [&](uint32_t slot, int R, int h) -> uint32_t {
            return is_v ? slot + uint32_t(R >> log2bs) * uint32_t(p.bs * 256) +
                              uint32_t(h * p.bs * 128) + uint32_t(R & (p.bs - 1)) * 128
                        : slot + uint32_t(h * L::kKVHalf) + uint32_t(R) * 128;
        };
        for (;;) {
            if (lane == 0)
                ok = wait_bounded(bar(kItemFull + (ic & 3)), (ic >> 2) & 1, abort_word);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            bool last;
            const Item I = slot_item(ring + (ic & 3), &last);
            mbar_arrive(bar(kItemEmpty + (ic & 3)));     // all 32 lanes arrive
            if (last) break;
            const int key_end = min(I.k_begin + I.n_tiles * kTileKeys, I.ctx);
            for (int jt = 0; jt < I.n_tiles; ++jt, ++tc) {
                // the table entries of kTableKeys keys at a time (the window of tile jt starts
                // at key sk)
                const int sk = I.k_begin + (jt & ~(kTableTiles - 1)) * kTileKeys;
                if ((jt & (kTableTiles - 1)) == 0) {
                    const int n_ent = min((min(sk + kTableKeys, key_end) - sk + p.bs - 1) >> log2bs,
                                          kMaxTableEntries);
                    const int32_t* trow =
                        p.block_table + int64_t(I.seq) * p.max_blocks + (sk >> log2bs);
                    __syncwarp();
                    for (int e = lane; e < n_ent; e += 32) {
                        int b = __ldg(trow + e);
                        if (b < 0 || b >= p.num_blocks) {
                            // out of range: the box lands outside the tensor and reads zeros
                            if (p.err && !is_v) atomicOr(p.err, PA_DEVERR_BLOCK);
                            b = -1;
                        }
                        tbl[e] = b;
                    }
                    __syncwarp();
                }
                const int st = tc % S;
                if (lane == 0 && tc >= S)
                    ok = wait_bounded(bar(empty_b + st), ((tc / S) - 1) & 1, abort_word);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const int kb = I.k_begin + jt * kTileKeys;
                const int key_hi = min(kb + kTileKeys, I.ctx);   // real keys end at ctx
                const int nblk = (key_hi - kb + p.bs - 1) >> log2bs;
                const uint32_t dst = slots + st * L::kKVTile;
                const int e0 = (kb - sk) >> log2bs;
                if constexpr (F8) {
                    // one box of bs rows x 128 code bytes per block, into the second halves
                    if (lane == 0) mbar_expect_tx(bar(full_b + st), uint32_t(nblk) * p.bs * 128);
                    __syncwarp();
                    for (int b = lane; b < nblk; b += 32)
                        tma_load_3d(row_base(dst, b * p.bs, 1), tmap, bar(full_b + st), 0, I.kvh,
                                    tbl[e0 + b] * p.bs);
                    continue;                   // the expander warp takes it from here
                }
                if (lane == 0)
                    mbar_expect_tx(bar(full_b + st), uint32_t(nblk) * p.bs * 128 * L::kChunks);
                __syncwarp();
                for (int j = lane; j < nblk * boxes_per_block; j += 32) {
                    const int b = j / boxes_per_block;
                    const int r = j - b * boxes_per_block;
                    const int z = tbl[e0 + b] * p.bs;
                    if (!is_v) {
                        // K: half r of the block, rows of the 128-key tile at 128-byte stride
                        tma_load_3d(dst + r * L::kKVHalf + b * p.bs * 128, tmap, bar(full_b + st),
                                    64 * r, I.kvh, z);
                    } else if constexpr (L::kChunks == 2) {
                        // V: both halves of the block, [half][row] inside the block
                        tma_load_4d(dst + b * p.bs * 256, tmap, bar(full_b + st), 0, z, 0, I.kvh);
                    } else {
                        tma_load_3d(dst + b * p.bs * 128, tmap, bar(full_b + st), 0, I.kvh, z);
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            ++ic;
        }
        if (lane == 0) {
            // never leave with copies in flight into this CTA's shared memory
            for (int t = max(0, tc - S); t < tc; ++t)
                wait_drain(bar(full_b + t % S), (t / S) & 1);
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ fp8 expanders (12, 14: K; 13, 15: V)
        // Walk the same tiles as the loaders: wait for a tile's codes to land, expand them to
        // f16 in place and publish the tile on its ready barrier (which the MMA, for K, or
        // the softmax, for V, waits for instead of the TMA barrier).
        if constexpr (F8) {
            const bool is_v = (warp & 1) != 0;
            const int half = (warp - 12) >> 1;           // rows 64 half .. 64 half + 63
            const volatile ItemSlot* ring =
                reinterpret_cast<const volatile ItemSlot*>(smem + L::kBar + kRingOff);
            const int log2bs = __ffs(p.bs) - 1;
            const int full_b = is_v ? kVFull : kKFull;
            const int ready_b = is_v ? kVReady : kKReady;
            const int S = is_v ? SV : SK;
            const uint32_t slots = sb + (is_v ? L::kV : L::kK);
            int tc = 0, ic = 0;
            int ok = 1;
            for (;;) {
                if (lane == 0)
                    ok = wait_bounded(bar(kItemFull + (ic & 3)), (ic >> 2) & 1, abort_word);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                bool last;
                const Item I = slot_item(ring + (ic & 3), &last);
                mbar_arrive(bar(kItemEmpty + (ic & 3)));     // all 32 lanes arrive
                if (last) break;
                for (int jt = 0; jt < I.n_tiles; ++jt, ++tc) {
                    const int st = tc % S;
                    if (lane == 0) ok = wait_bounded(bar(full_b + st), (tc / S) & 1, abort_word);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    const int kb = I.k_begin + jt * kTileKeys;
                    const int key_hi = min(kb + kTileKeys, I.ctx);
                    const int rows = ((key_hi - kb + p.bs - 1) >> log2bs) * p.bs;
                    const uint32_t slot = slots + st * L::kKVTile;
                    const int r_end = min(rows, 64 * half + 64);
                    if (is_v)
                        expand_codes<true>(slot, 64 * half, r_end, p.bs, log2bs, lane);
                    else
                        expand_codes<false>(slot, 64 * half, r_end, p.bs, log2bs, lane);
                    // generic-proxy writes, read by the MMA through the async proxy
                    fence_proxy_async();
                    __syncwarp();
                    mbar_arrive(bar(ready_b + st));             // all 32 lanes arrive
                }
                if (!ok) break;
                ++ic;
            }
        }
    } else {
        // ------------------------------------------------------------ softmax warps 0-7
        // Warp w reads TMEM sub-partition w % 4 and takes its 16-lane half w / 4: rows
        // r0 + rs and r0 + rs + 8 of the tile (r0 = 32 (w % 4) + 16 (w / 4), rs = lane / 4).
        const int tid = threadIdx.x;              // 0..255
        const int r0 = 32 * (warp & 3) + 16 * (warp >> 2);
        const uint32_t lanes = uint32_t(r0) << 16;
        const int q4 = lane & 3;
        const int rs = lane >> 2;
        const float c = p.c;
        const volatile ItemSlot* ring =
            reinterpret_cast<const volatile ItemSlot*>(smem + L::kBar + kRingOff);
        int tc = 0, ic = 0, sg = 0;       // tiles, items and splits seen
        int ng = 0;                       // GROUP items whose state has been saved
        bool ok = true;
        // the wait-timeout test: a wait that nothing completes runs out, and every role leaves
        // through the same path as after any other wait that ran out
        if (p.never_ns) ok = wait_bounded(bar(kNever), 0, abort_word, p.never_ns);
        for (; ok;) {
            if (!(ok = wait_bounded(bar(kItemFull + (ic & 3)), (ic >> 2) & 1, abort_word))) break;
            bool last;
            const Item I = slot_item(ring + (ic & 3), &last);
            mbar_arrive(bar(kItemEmpty + (ic & 3)));
            if (last) break;
            const bool on = r0 < I.rows_valid;    // warp-uniform: the warp holds a valid row
            Rows2 R;
            Fold2 F;
            // a RESUME item starts inside split 0, at tile tile0 (0 for every other item)
            const int jt0 = I.tile0;
            if (jt0 > 0) {
                // the state its GROUP item saved (that item is earlier on this CTA's list; its
                // O buffer was released by these warps' own epilogue two splits ago)
                if (ng == 0) {
                    if (tid == 0 && p.err) atomicOr(p.err, PA_DEVERR_META);
                } else if (!(ok = wait_bounded(bar(kSaved), (ng - 1) & 1, abort_word))) {
                    break;
                }
                if (on)
                    R = restore_half<D>(p.ws_acc, p.ws_ml, p.g, p.max_splits, p.Hq,
                                        tmem + kTmemO + (sg & 1) * 128 + lanes, r0, rs, q4,
                                        I.rows_valid, I.q_start, I.kvh, I.pos0);
            }
            for (int jt = 0; jt < I.n_tiles; ++jt, ++tc) {
                // every split starts afresh, exactly as an item of that split alone would
                const int jin = (jt0 + jt) & (kSplitTiles - 1);
                if (jin == 0) rows_init(R, r0, rs, I.rows_valid, I.pos0, p.g);
                const int ob = sg & 1;
                const uint32_t tm_o = tmem + kTmemO + ob * 128 + lanes;
                if (!(ok = wait_bounded(bar(kSFull + (tc & (SK - 1))), (tc >> kLog2SK) & 1,
                                        abort_word)))
                    break;
                tc_fence_after();
                const int kb = I.k_begin + jt * kTileKeys;
                float alpha[2] = {1.f, 1.f};
                if (on)
                    softmax_half<F8>(tmem + (tc & 1) * 128 + lanes, r0, q4, I.rows_valid, kb, c, R,
                                     alpha);
                // O belongs to the previous tile's PV until it has finished: rescale only then,
                // and only in warps where some row's running maximum moved
                const bool need = alpha[0] != 1.f || alpha[1] != 1.f;
                if (jin > 0 && __any_sync(0xffffffffu, need)) {
                    if (!(ok = wait_bounded(bar(kPVDone + (tc - 1) % SV), ((tc - 1) / SV) & 1,
                                            abort_word)))
                        break;
                    tc_fence_after();
                    rescale_half<D>(tm_o, alpha);
                }
                tmem_wait_st();
                // V of the tile has landed before P is published (the PV issue relies on it);
                // keys at or beyond ctx are stale or were never loaded: give them zero values
                // so that their (zero) probabilities contribute exact zeros
                if (!(ok = wait_bounded(bar(kVUse + tc % SV), (tc / SV) & 1, abort_word))) break;
                if (kb + kTileKeys > I.ctx) {
                    zero_v_tail<D>(sb + L::kV + (tc % SV) * L::kKVTile, kb, I.ctx, p.bs, tid, 256);
                    // the zeros were written through the generic proxy and the PV MMA reads
                    // them through the async proxy: only these tiles need the proxy fence
                    fence_proxy_async();
                }
                tc_fence_before();
                mbar_arrive(bar(kPFull + (tc & 1)));            // all 256 softmax threads arrive
                if (jin != kSplitTiles - 1 && jt != I.n_tiles - 1) continue;
                // ------------------------------------------------------ end of a split
                const int js = (jt0 + jt) / kSplitTiles;   // split of the item (0 for a decode's)
                ++sg;
                if (I.n_splits > 1 && js == 0) {
                    // split 0's O stays where it is as the running result: nothing to wait for
#pragma unroll
                    for (int sr = 0; sr < 2; ++sr) {
                        F.M[sr] = R.m[sr];
                        F.L[sr] = R.l[sr];
                    }
                    continue;
                }
                if (!(ok = wait_bounded(bar(kPVDone + tc % SV), (tc / SV) & 1, abort_word)))
                    break;
                tc_fence_after();
                if (I.n_splits > 1) {
                    const bool fin = js == I.n_splits - 1;
                    const uint32_t tm_a = tmem + kTmemO + (ob ^ 1) * 128 + lanes;
                    if (on)
                        fold_half<D>(p, tm_a, tm_o, r0, rs, q4, I.rows_valid, I.q_start, I.kvh,
                                     js, fin, R, F);
                    tc_fence_before();
                    mbar_arrive(bar(kOFree + (ob ^ 1)));     // the previous running result
                    if (fin) mbar_arrive(bar(kOFree + ob));
                } else if (!on) {
                    tc_fence_before();
                    mbar_arrive(bar(kOFree + ob));
                } else {
                    uint32_t o[D / 2];
                    if constexpr (D == 128) tmem_ld_16x256b_x16(tm_o, o);
                    else tmem_ld_16x256b_x8(tm_o, o);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(bar(kOFree + ob));       // O is in registers: its buffer is free
                    store_half<D>(p, o, r0, rs, q4, I.rows_valid, I.q_start, I.kvh, I.split, R,
                                  I.kind == PA_ITEM_GROUP);
                }
                if (I.kind == PA_ITEM_GROUP) {
                    // the saved state is published to the RESUME items (other threads of these
                    // warps restore it)
                    __threadfence_block();
                    mbar_arrive(bar(kSaved));
                    ++ng;
                }
            }
            if (!ok) break;
            ++ic;
        }
    }
    if (*abort_word && threadIdx.x == 0 && p.err) atomicOr(p.err, PA_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------- fixed-order split combine
// For every (decode row, q head) whose row spans more than one split: fold the partials of
// splits 0, 1, ... in ascending order, starting from split 0's (m, l, acc) as they are:
//   M' = max(M, m_s), a = 2^((M - M') c), b = 2^((m_s - M') c),
//   L = L a + l_s b, ACC = ACC a + acc_s b;  out = bf16_rne(ACC * (rcp_rn(L) * v_scale))
// (v_scale is 1 for a bf16 cache, so that product is rcp_rn(L) exactly).
// A row with one split is finished by the attention kernel with the same two roundings, and
// so is every row of a sequence with several query rows, whose item folds its own splits in
// this order (fold_half). One thread per (sequence, q head, 4 columns); sequences with other
// than one query row return at once. The partials of up to kBatch splits are loaded before
// they are folded, so a row costs about nsplit / kBatch memory round trips. Launched
// as a programmatic dependent of the attention kernel (its launch overlaps the attention
// tail); griddepcontrol.wait holds every thread until that grid has completed and its
// writes are visible.
template <int D>
__global__ void __launch_bounds__(256)
    combine_kernel(const float* __restrict__ ws_acc, const float* __restrict__ ws_ml,
                   const int32_t* __restrict__ cu, const int32_t* __restrict__ ctx, int32_t B,
                   int32_t T, int32_t Hq, int32_t max_splits, float c, float v_scale,
                   __nv_bfloat16* __restrict__ out) {
    constexpr int kCols = 4;                  // columns per thread (one float4)
    constexpr int kUnits = D / kCols;         // threads per (row, q head)
    constexpr int kBatch = 8;                 // splits loaded ahead of their fold
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t n = int64_t(B) * Hq * kUnits;
    const int64_t u = int64_t(blockIdx.x) * 256 + threadIdx.x;
    if (u >= n) return;
    const int64_t w = u / kUnits;
    const int col = int(u % kUnits) * kCols;
    const int s = int(w / Hq);
    const int head = int(w % Hq);
    const int64_t tok = __ldg(cu + s);
    // metadata the attention kernel rejects (a row outside [0, T)) is skipped here too, so
    // that no partial or output outside the caller's buffers is touched
    if (__ldg(cu + s + 1) - tok != 1 || tok < 0 || tok >= T) return;
    const int pos = __ldg(ctx + s) - 1;
    if (pos < 0) return;                      // inconsistent metadata: flagged by the kernel
    const int nsp = pos / kSplit + 1;
    if (nsp == 1 || nsp > max_splits) return;
    const int64_t base = tok * max_splits;
    const float2* ml = reinterpret_cast<const float2*>(ws_ml);
    float M, Lsum, acc[kCols];
    {
        const int64_t slot = base * Hq + head;
        const float2 m0 = ml[slot];
        const float4 a0 = *reinterpret_cast<const float4*>(ws_acc + slot * D + col);
        M = m0.x;
        Lsum = m0.y;
        acc[0] = a0.x;
        acc[1] = a0.y;
        acc[2] = a0.z;
        acc[3] = a0.w;
    }
    for (int s0 = 1; s0 < nsp; s0 += kBatch) {
        float2 ms[kBatch];
        float4 as[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (s0 + j < nsp) {
                const int64_t slot = (base + s0 + j) * Hq + head;
                ms[j] = ml[slot];
                as[j] = *reinterpret_cast<const float4*>(ws_acc + slot * D + col);
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (s0 + j >= nsp) break;
            const float mn = fmaxf(M, ms[j].x);
            const float fa = M == mn ? 1.f : ex2(__fmul_rn(__fsub_rn(M, mn), c));
            const float fb = ms[j].x == mn ? 1.f : ex2(__fmul_rn(__fsub_rn(ms[j].x, mn), c));
            Lsum = __fadd_rn(__fmul_rn(Lsum, fa), __fmul_rn(ms[j].y, fb));
            const float av[kCols] = {as[j].x, as[j].y, as[j].z, as[j].w};
#pragma unroll
            for (int e = 0; e < kCols; ++e)
                acc[e] = __fadd_rn(__fmul_rn(acc[e], fa), __fmul_rn(av[e], fb));
            M = mn;
        }
    }
    const float inv = __fmul_rn(__frcp_rn(Lsum), v_scale);
    __nv_bfloat16* dst = out + (tok * Hq + head) * D + col;
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(pack_bf16(__fmul_rn(acc[0], inv), __fmul_rn(acc[1], inv)),
                   pack_bf16(__fmul_rn(acc[2], inv), __fmul_rn(acc[3], inv)));
}

// ------------------------------------------------------------------------- host side

// The driver's tensor-map encoder, looked up once per process (a function-local static is
// initialised exactly once even when several host threads call this at the same time).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        return PFN_cuTensorMapEncodeTiled_v12000(nullptr);
    }();
    return fn;
}

// A bf16 3-D tensor {D, heads, rows} with 128-byte swizzled boxes {64, box_heads, box_rows}.
int32_t make_map(CUtensorMap* m, const void* base, int D, int heads, int64_t rows,
                 int box_heads, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return PA_ERR_CUDA;
    const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(heads), cuuint64_t(rows)};
    const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(heads) * D * 2};
    const cuuint32_t box[3] = {64, cuuint32_t(box_heads), cuuint32_t(box_rows)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// An fp8 pool as {D, heads, rows} bytes: one box is one block of one KV head, bs rows of D
// code bytes, unswizzled (the loader expands it in shared memory).
int32_t make_map_codes(CUtensorMap* m, const void* base, int D, int heads, int64_t rows,
                       int box_rows) {
    auto fn = encode_fn();
    if (!fn) return PA_ERR_CUDA;
    const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(heads), cuuint64_t(rows)};
    const cuuint64_t strides[2] = {cuuint64_t(D), cuuint64_t(heads) * D};
    const cuuint32_t box[3] = {cuuint32_t(D), 1, cuuint32_t(box_rows)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

struct Maps {
    CUtensorMap k, v, q1, qn;
};

// K/V pools as {D, Hkv, num_blocks * block_size}: one box is one block of one KV head and one
// 64-column chunk. q as {D, Hq, T}: a decode item's box is its g heads of one token, a prefill
// item's box is g heads of 128/g tokens (rows past the item are not used; past T they read 0).
int32_t make_maps(Maps* m, const void* q, const void* k_pool, const void* v_pool, int32_t T,
                  const pa_shape* s, bool fp8) {
    const int D = s->head_dim;
    const int g = s->num_q_heads / s->num_kv_heads;
    const int64_t rows = int64_t(s->num_blocks) * s->block_size;
    int32_t st;
    if (fp8) {
        if ((st = make_map_codes(&m->k, k_pool, D, s->num_kv_heads, rows, s->block_size)))
            return st;
        if ((st = make_map_codes(&m->v, v_pool, D, s->num_kv_heads, rows, s->block_size)))
            return st;
    } else if ((st = make_map(&m->k, k_pool, D, s->num_kv_heads, rows, 1, s->block_size))) {
        return st;
    }
    if (fp8) {
        // both code maps are built above
    } else if (D == 128) {
        // {64, rows, half, head}: one box holds both 64-column halves of one block, halves
        // outermost, so that each half's rows are contiguous in shared memory
        auto fn = encode_fn();
        if (!fn) return PA_ERR_CUDA;
        const cuuint64_t dims[4] = {64, cuuint64_t(rows), 2, cuuint64_t(s->num_kv_heads)};
        const cuuint64_t strides[3] = {cuuint64_t(s->num_kv_heads) * D * 2, 128, cuuint64_t(D) * 2};
        const cuuint32_t box[4] = {64, cuuint32_t(s->block_size), 2, 1};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        if (fn(&m->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(v_pool), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PA_ERR_CUDA;
    } else if ((st = make_map(&m->v, v_pool, D, s->num_kv_heads, rows, 1, s->block_size))) {
        return st;
    }
    if ((st = make_map(&m->q1, q, D, s->num_q_heads, T, g, 1))) return st;
    return make_map(&m->qn, q, D, s->num_q_heads, T, g, kRows / g);
}

constexpr int kMaxDevices = 64;

// Raises the kernel's dynamic shared-memory limit once per device. Several host threads (one
// per GPU, say) may get here at once: the flags are atomic, and the attribute call is
// idempotent, so two threads that both find a flag clear both set the same value.
template <int D, bool F8>
int32_t ensure_smem_attr(int dev) {
    static std::atomic<bool> raised[kMaxDevices];     // zero-initialised: not raised yet
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_INVALID;
    if (raised[dev].load(std::memory_order_acquire)) return PA_OK;
    const int32_t st = note_cuda(cudaFuncSetAttribute(
        paged_attn_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<D>::kAlloc));
    if (st) return st;
    raised[dev].store(true, std::memory_order_release);
    return PA_OK;
}

template <int D, bool F8>
int32_t launch(const Maps& maps, const Params& prm, int32_t max_ctx, cudaStream_t stream) {
    int dev = 0;
    int32_t st = note_cuda(cudaGetDevice(&dev));
    if (st) return st;
    if ((st = ensure_smem_attr<D, F8>(dev))) return st;
    const int grid = std::min(prm.n_items, PA_PLAN_CTAS);      // one CTA per list of the plan
    // Both kernels are programmatic dependents of what precedes them on the stream: each
    // launches while its predecessor drains and waits (griddepcontrol.wait) before it reads
    // anything.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kThreadsFor<F8>);
    cfg.dynamicSmemBytes = Layout<D>::kAlloc;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    st = note_cuda(cudaLaunchKernelEx(&cfg, paged_attn_kernel<D, F8>, maps.k, maps.v, maps.q1,
                                      maps.qn, prm));
    if (st) return st;
    if (max_ctx > kSplit) {
        const int64_t threads = int64_t(prm.B) * prm.Hq * (D / 4);
        cfg.gridDim = dim3(unsigned((threads + 255) / 256));
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        st = note_cuda(cudaLaunchKernelEx(&cfg, combine_kernel<D>, (const float*)prm.ws_acc,
                                          (const float*)prm.ws_ml, prm.cu, prm.ctx, prm.B, prm.T,
                                          prm.Hq, prm.max_splits, prm.c, prm.v_scale, prm.out));
    }
    return st;
}

// Host checks and parameter set-up shared by both step entry points.
int32_t prepare_step(const void* q, const void* k_pool, const void* v_pool,
                     const int32_t* block_table, int32_t max_blocks, const int32_t* cu_seqlens_q,
                     const int32_t* ctx_lens, int32_t B, int32_t T, int32_t max_ctx,
                     const pa_work_item* items, int32_t n_items, void* out,
                     const pa_shape* shape, int32_t* err_flag, Maps* maps, Params* prm,
                     bool fp8 = false) {
    int32_t st = check_shape(shape);
    if (st) return st;
    if (B < 0 || T < 0 || n_items < 0 || max_ctx < 0 || max_blocks < 0) return PA_ERR_INVALID;
    if (!q || !k_pool || !v_pool || !block_table || !cu_seqlens_q || !ctx_lens || !items || !out)
        return PA_ERR_INVALID;
    if (int64_t(shape->num_blocks) * shape->block_size > INT32_MAX) return PA_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool) |
         reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15)
        return PA_ERR_INVALID;
    if ((st = make_maps(maps, q, k_pool, v_pool, T, shape, fp8))) return st;
    const int D = shape->head_dim;
    prm->k_pool = static_cast<const __nv_bfloat16*>(k_pool);
    prm->v_pool = static_cast<const __nv_bfloat16*>(v_pool);
    prm->block_table = block_table;
    prm->cu = cu_seqlens_q;
    prm->ctx = ctx_lens;
    prm->items = items;
    prm->ws_acc = nullptr;
    prm->ws_ml = nullptr;
    prm->out = static_cast<__nv_bfloat16*>(out);
    prm->err = err_flag;
    prm->n_items = n_items;
    prm->B = B;
    prm->T = T;
    prm->max_blocks = max_blocks;
    prm->max_splits = int((int64_t(max_ctx) + kSplit - 1) / kSplit);
    prm->Hq = shape->num_q_heads;
    prm->Hkv = shape->num_kv_heads;
    prm->g = shape->num_q_heads / shape->num_kv_heads;
    prm->bs = shape->block_size;
    prm->num_blocks = shape->num_blocks;
    prm->c = float(1.4426950408889634 / std::sqrt(double(D)));
    prm->v_scale = 1.f;
    prm->never_ns = 0;
    return PA_OK;
}

// Workspace: acc [T][max_splits][Hq][D] fp32, then (m, l) [T][max_splits][Hq][2] fp32.
void point_workspace(Params* prm, float* ws, int32_t T, int32_t Hq, int D) {
    prm->ws_acc = ws;
    prm->ws_ml = ws ? ws + size_t(T) * prm->max_splits * Hq * D : nullptr;
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
    if (max_ctx > kSplit && (!workspace || ws_bytes < pa_workspace_bytes(shape, T, max_ctx)))
        return PA_ERR_WORKSPACE;
    // the partials are stored and loaded as 8- and 16-byte vectors
    if (max_ctx > kSplit && (reinterpret_cast<uintptr_t>(workspace) & 15)) return PA_ERR_INVALID;
    Maps maps;
    Params prm;
    if ((st = prepare_step(q, k_pool, v_pool, block_table, max_blocks, cu_seqlens_q, ctx_lens, B,
                           T, max_ctx, items, n_items, out, shape, err_flag, &maps, &prm)))
        return st;
    point_workspace(&prm, static_cast<float*>(workspace), T, shape->num_q_heads, shape->head_dim);
    if (shape->head_dim == 128) return launch<128, false>(maps, prm, max_ctx, stream);
    return launch<64, false>(maps, prm, max_ctx, stream);
}

// The wait-timeout test: paged_attention_step with the softmax role first waiting, for at most
// never_ns, on a barrier that nothing completes (see pagedattn.h).
extern "C" int32_t paged_attention_step_wait_test(
    const void* q, const void* k_pool, const void* v_pool, const int32_t* block_table,
    int32_t max_blocks, const int32_t* cu_seqlens_q, const int32_t* ctx_lens, int32_t B,
    int32_t T, int32_t max_ctx, const pa_work_item* items, int32_t n_items, void* workspace,
    size_t ws_bytes, void* out, const pa_shape* shape, int32_t* err_flag,
    uint64_t never_ns, pa_stream_t stream) {
    int32_t st = check_shape(shape);
    if (st) return st;
    if (B < 0 || T < 0 || n_items < 0 || max_ctx < 0 || max_blocks < 0) return PA_ERR_INVALID;
    if (never_ns == 0 || never_ns > kWaitLimitNs) return PA_ERR_INVALID;
    if (T == 0 || n_items == 0) return PA_OK;
    if (max_ctx > kSplit && (!workspace || ws_bytes < pa_workspace_bytes(shape, T, max_ctx)))
        return PA_ERR_WORKSPACE;
    if (max_ctx > kSplit && (reinterpret_cast<uintptr_t>(workspace) & 15)) return PA_ERR_INVALID;
    Maps maps;
    Params prm;
    if ((st = prepare_step(q, k_pool, v_pool, block_table, max_blocks, cu_seqlens_q, ctx_lens, B,
                           T, max_ctx, items, n_items, out, shape, err_flag, &maps, &prm)))
        return st;
    prm.never_ns = never_ns;
    point_workspace(&prm, static_cast<float*>(workspace), T, shape->num_q_heads, shape->head_dim);
    if (shape->head_dim == 128) return launch<128, false>(maps, prm, max_ctx, stream);
    return launch<64, false>(maps, prm, max_ctx, stream);
}

// FP8 KV cache: the same step over float8_e4m3fn pools with per-tensor scales. The K scale
// joins the softmax constant (scores are taken on the codes' values), the V scale the final
// factor of every row: out = bf16(O * (rcp(l) * v_scale)).
extern "C" int32_t paged_attention_step_fp8(const void* q, const void* k_pool, const void* v_pool,
                                            const int32_t* block_table, int32_t max_blocks,
                                            const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                                            int32_t B, int32_t T, int32_t max_ctx,
                                            const pa_work_item* items, int32_t n_items,
                                            float k_scale, float v_scale, void* workspace,
                                            size_t ws_bytes, void* out, const pa_shape* shape,
                                            int32_t* err_flag, pa_stream_t stream) {
    int32_t st = check_shape(shape);
    if (st) return st;
    if (shape->head_dim != 128) return PA_ERR_SHAPE;
    if (B < 0 || T < 0 || n_items < 0 || max_ctx < 0 || max_blocks < 0) return PA_ERR_INVALID;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !(k_scale < INFINITY) || !(v_scale < INFINITY))
        return PA_ERR_INVALID;
    if (T == 0 || n_items == 0) return PA_OK;
    if (max_ctx > kSplit && (!workspace || ws_bytes < pa_workspace_bytes(shape, T, max_ctx)))
        return PA_ERR_WORKSPACE;
    if (max_ctx > kSplit && (reinterpret_cast<uintptr_t>(workspace) & 15)) return PA_ERR_INVALID;
    Maps maps;
    Params prm;
    if ((st = prepare_step(q, k_pool, v_pool, block_table, max_blocks, cu_seqlens_q, ctx_lens, B,
                           T, max_ctx, items, n_items, out, shape, err_flag, &maps, &prm, true)))
        return st;
    prm.c = prm.c * k_scale;
    prm.v_scale = v_scale;
    point_workspace(&prm, static_cast<float*>(workspace), T, shape->num_q_heads, shape->head_dim);
    return launch<128, true>(maps, prm, max_ctx, stream);
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
    // the partials of this step must fit the fixed array; nothing is launched otherwise
    if (max_ctx > kSplit && pa_workspace_bytes(shape, T, max_ctx) > PA_STATIC_SCRATCH_BYTES)
        return PA_ERR_WORKSPACE;
    Maps maps;
    Params prm;
    if ((st = prepare_step(q, k_pool, v_pool, block_table, max_blocks, cu_seqlens_q, ctx_lens, B,
                           T, max_ctx, items, n_items, out, shape, err_flag, &maps, &prm)))
        return st;
    float* scratch = nullptr;
    if ((st = static_scratch_for_current_device(&scratch))) return st;
    point_workspace(&prm, scratch, T, shape->num_q_heads, shape->head_dim);
    if (shape->head_dim == 128) return launch<128, false>(maps, prm, max_ctx, stream);
    return launch<64, false>(maps, prm, max_ctx, stream);
}
