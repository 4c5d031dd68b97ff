// Causal chunked prefill over the paged pool on GB300's fifth-generation
// tensor cores (tcgen05 with accumulators in tensor memory).
//
// What is computed follows the varlen read of the vLLM book's chapter 4
// ("第4章 PagedAttention：虚拟内存的启示", §4.5 step 2: the backend hands
// the cache, cu_seqlens_q, seqused_k and the block table to one call): a
// chunk of q_len query tokens is the last q_len of the sequence's seq_len
// cached tokens, query i sits at position p = seq_len - q_len + i, and it
// attends to tokens 0..p through the block table, with the online softmax
// of §4.6.
//
// How it is computed:
//  * Work units. A unit is two adjacent 128-row query tiles (A and B) of
//    one (sequence, kv head, head tile); rows are (query head of the group,
//    query token) pairs, so the heads sharing a kv head, and both tiles,
//    share every K/V tile. One persistent CTA per SM takes units from a
//    per-launch counter (warp 11, which also loads each unit's Q) and hands
//    them to every role through a small ring; TMA rings and barrier phases
//    run on across units.
//  * Few units (a few long sequences with short chunks). With at most four
//    units per SM and a workspace, the CTAs instead take equal contiguous
//    shares of all units' K/V tiles (stream-K), so a unit's range may be
//    cut into pieces on several SMs; a piece stores its partial softmax
//    state, and paged_prefill_merge_kernel combines the pieces of each unit
//    with the §4.6 rule in a fixed order.
//  * Loads. Warp 8 brings the K tiles and warp 10 the V tiles by TMA
//    (16-token boxes through the block table, 128-byte swizzle) into rings
//    of two K and three V stages (a V stage is released as soon as its last
//    P V is issued). With an FP8 cache (two and two), warps 12-15 instead
//    bring the codes into staging buffers and widen them exactly into fp16
//    ring stages (two K stages then); the MMAs then run in fp16, and bf16
//    queries are moved to fp16 row by row under a power-of-two scale that
//    joins the row's score factor.
//  * Tensor memory holds S_A, S_B, O_A and O_B; P is written over the first
//    64 columns of its S as 16-bit pairs. One thread of warp 9 issues, per
//    K/V tile j, O_A += P_A V_j, S_A(j+1), O_B += P_B V_j, S_B(j+1)
//    (tcgen05, P read from tensor memory, V as an MN-major operand), so one
//    tile's matrix work overlaps the other tile's softmax.
//  * Softmax. Warpgroup x owns tile x, a full row per thread: read S, mask
//    causally, row maximum as scale x raw extremum, P = 2^(s scale - ref)
//    rounded to the element type (the reference maximum moves only when a
//    score exceeds it by 2^8, so O is rarely rescaled), row sum of the
//    rounded values, P into tensor memory. At the unit's end, O / l.
//  * Every wait is bounded; K/V rows past a sequence's end (padding slots,
//    possibly NaN) are zeroed before P V reads them.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "../../include/pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__device__ int g_prefill_error;  // PA_DEVERR_* bits of the prefill kernels

// Work-unit counters of in-flight prefill launches: {next unit, CTAs done}
// per slot; a launch takes slot (launch number % 64), the last CTA to finish
// puts both back to 0.
constexpr int kSchedSlots = 64;
__device__ int g_prefill_sched[kSchedSlots][2];

// Stream-K launches (few work units): at most this many units.
constexpr int kMaxSplitUnits = 1024;
constexpr int kMergeRowsPerThread = 4;  // rows one merge thread combines

namespace {

__device__ __forceinline__ void prefill_raise(int bit) { atomicOr(&g_prefill_error, bit); }

// ------------------------------------------------------------- tcgen05 PTX

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B both fp16
// or both bf16, A K-major, B K-major or MN-major, M x N.
__device__ __forceinline__ uint32_t instr_desc(int m, int n, bool bf16, bool b_mn)
{
    uint32_t d = 1u << 4;
    d |= (bf16 ? 1u : 0u) << 7;
    d |= (bf16 ? 1u : 0u) << 10;
    d |= (b_mn ? 1u : 0u) << 16;
    d |= (uint32_t)(n >> 3) << 17;
    d |= (uint32_t)(m >> 4) << 24;
    return d;
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective);
// the registers are valid after tc_wait_ld().
__device__ __forceinline__ void tc_ld32_async(uint32_t taddr, uint32_t *r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The same, waited for and converted.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float *v)
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const float *v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]),
        "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]),
        "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]),
        "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
}

// O += A B with A read from TMEM (32-bit columns holding two 16-bit
// elements, the lower-indexed one in the low half) and B from shared memory.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Two E4M3 codes (the low / high 16 bits of x, the lower byte to the lower
// half) to an fp16 pair; exact, every E4M3 value is an fp16 value.
__device__ __forceinline__ uint32_t e4m3_pair_lo(uint32_t x)
{
    uint32_t d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(d) : "r"(x));
    return d;
}

__device__ __forceinline__ uint32_t e4m3_pair_hi(uint32_t x)
{
    uint32_t d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, hi;\n\t}" : "=r"(d) : "r"(x));
    return d;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Three-input maximum / minimum.
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float min3(float a, float b, float c)
{
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// acc + the two 16-bit elements of a packed pair (low half first), each added
// exactly as fp32 then rounded: mixed-precision adds, no unpacking.
template <bool BF16>
__device__ __forceinline__ float add_pair(float acc, uint32_t w)
{
    const unsigned short lo = (unsigned short)(w & 0xFFFFu), hi = (unsigned short)(w >> 16);
    if constexpr (BF16) {
        asm("add.rn.f32.bf16 %0, %1, %0;" : "+f"(acc) : "h"(lo));
        asm("add.rn.f32.bf16 %0, %1, %0;" : "+f"(acc) : "h"(hi));
    } else {
        asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(acc) : "h"(lo));
        asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(acc) : "h"(hi));
    }
    return acc;
}

// Two fp32 lanes at once (the packed .f32x2 forms: one instruction each).
__device__ __forceinline__ uint64_t pk2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpk2(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// 2^x0, 2^x1 on the FMA pipe, without the MUFU unit that ex2 uses: x = j + f
// with j = round(x) (adding and subtracting 1.5 * 2^23 rounds to an integer
// in fp32 for |x| < 2^22) and f in [-1/2, 1/2] exact, then p(f) ~ 2^f by the
// minimax polynomial of degree DEG (coefficients from a Remez exchange fit of
// the relative error, printed by paged_kv_cache_120_gb300/exp2_poly.py; max
// relative error 7.5e-5 at degree 3, 2.7e-6 at degree 4), then j added to
// p's exponent field. Inputs below -126 are clamped there (2^-126 or less
// rounds to zero or to a negligible subnormal in the 16-bit P); NaN stays
// NaN (max.NaN keeps it, and the exponent add leaves NaN bits NaN).
template <int DEG>
__device__ __forceinline__ void exp2_poly2(uint64_t x2, float &y0, float &y1)
{
    float x0, x1;
    unpk2(x2, x0, x1);
    asm("max.NaN.f32 %0, %0, 0fC2FC0000;" : "+f"(x0));  // -126
    asm("max.NaN.f32 %0, %0, 0fC2FC0000;" : "+f"(x1));
    const uint64_t xv = pk2(x0, x1);
    const uint64_t magic = pk2(12582912.f, 12582912.f), nmagic = pk2(-12582912.f, -12582912.f);
    const uint64_t j = add2(xv, magic);           // round(x) in the low mantissa bits
    const uint64_t t = add2(j, nmagic);           // round(x) as a float
    uint64_t f;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(f) : "l"(xv), "l"(t));
    uint64_t p;
    if constexpr (DEG == 4) {
        p = fma2(pk2(0x1.3997d6p-7f, 0x1.3997d6p-7f), f, pk2(0x1.ca1440p-5f, 0x1.ca1440p-5f));
        p = fma2(p, f, pk2(0x1.ec06dap-3f, 0x1.ec06dap-3f));
        p = fma2(p, f, pk2(0x1.62e0dcp-1f, 0x1.62e0dcp-1f));
        p = fma2(p, f, pk2(0x1.ffffe8p-1f, 0x1.ffffe8p-1f));
    } else {
        static_assert(DEG == 3, "degree 3 or 4");
        p = fma2(pk2(0x1.c3f760p-5f, 0x1.c3f760p-5f), f, pk2(0x1.f0de1ap-3f, 0x1.f0de1ap-3f));
        p = fma2(p, f, pk2(0x1.62f31ap-1f, 0x1.62f31ap-1f));
        p = fma2(p, f, pk2(0x1.fff692p-1f, 0x1.fff692p-1f));
    }
    float p0, p1, j0, j1;
    unpk2(p, p0, p1);
    unpk2(j, j0, j1);
    y0 = __uint_as_float(__float_as_uint(p0) + (__float_as_uint(j0) << 23));
    y1 = __uint_as_float(__float_as_uint(p1) + (__float_as_uint(j1) << 23));
}

// 32 consecutive 32-bit columns of this thread's TMEM lane from raw words.
__device__ __forceinline__ void tc_st32u(uint32_t taddr, const uint32_t *v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// ----------------------------------------------------------------- layout

constexpr int kD = 128;                    // largest head size built (64 and 128)
constexpr int kM = 128;                    // query rows per tile (TMEM lanes)
constexpr int kN = 128;                    // cached tokens per K/V tile
constexpr int kChunkBytes = 128 * 128;     // a 64-column, 128-row swizzled chunk: 16 KB
constexpr int kTileBytes = 2 * kChunkBytes;  // a 128 x 128 16-bit operand: 32 KB
constexpr int kBoxTokens = 16;             // tokens per K/V TMA box (block_size is a multiple)
// Warps 0-3 softmax A, 4-7 softmax B, 8 K, 9 MMA, 10 V, 11 Q; with an FP8
// cache also 12-15, which widen the codes (8 and 10 then stay idle).
constexpr int kThreads16 = 384, kThreads8 = 512;
__host__ __device__ constexpr int threads_for(bool fp8) { return fp8 ? kThreads8 : kThreads16; }
constexpr int kWarpK = 8, kWarpMMA = 9, kWarpV = 10, kWarpQ = 11;
// K ring (a stage is freed when both tiles' S = Q K^T are done) and V ring
// (freed when both tiles' O += P V are done). The V tile is needed first
// in a K/V step and K one half step later, so V gets the deeper ring: 2 K
// and 3 V stages with a 16-bit cache, 2 and 2 with an FP8 cache (whose
// staging buffers take the rest of shared memory).
constexpr int kKStagesMax = 2, kVStagesMax = 3;
constexpr int kKStages16 = 2, kKStages8 = 2;
constexpr int kVStages16 = 3, kVStages8 = 2;
constexpr int kOffQ = 0;                   // Q of tile A, then of tile B
constexpr int kOffK = 2 * kTileBytes;
constexpr int kStageBytes8 = 128 * 128;    // an FP8 K or V tile as loaded, before widening: 16 KB
// 16-bit cache: Q 64 KB, K 2 x 32, V 3 x 32. FP8 cache: Q 64, K 2 x 32, V 2 x 32,
// then one FP8 staging tile each for K and V (16 KB each). Both 224 KB.
constexpr int kSmemBytes = 2 * kTileBytes + 5 * kTileBytes + 1024;  // + align slack
static_assert((kKStages16 + kVStages16) * kTileBytes <= 5 * kTileBytes &&
              (kKStages8 + kVStages8) * kTileBytes + 2 * kStageBytes8 <= 5 * kTileBytes, "shared memory plan");
constexpr uint32_t kTmemCols = 512;        // S/P of tiles A and B, then O of A and B, 128 columns each
constexpr float kRescaleLog2 = 8.f;        // reference-maximum slack (base 2)
// If > 0: in a full score tile, every kPolyEvery-th pair of exponentials is
// computed by a polynomial on the FMA pipe instead of the MUFU unit. Off: on
// GB300 the softmax is bound by instruction latency, not by the MUFU unit,
// and the extra instructions cost more than they relieve (measured: every
// 3rd pair made the Llama-2-13B-shaped prefill 12% slower).
#ifndef PA_PREFILL_POLY_EVERY
#define PA_PREFILL_POLY_EVERY 0
#endif
constexpr int kPolyEvery = PA_PREFILL_POLY_EVERY;
constexpr int kUnitSlots = 4;              // ring of unit indices handed from the scheduler to every role
// Unit consumers (one arrival each): K, V and MMA warps and the 8 softmax
// warps; with an FP8 cache the 4 widening warps instead of K and V.
__host__ __device__ constexpr int unit_consumers(bool fp8) { return fp8 ? 13 : 11; }
// Registers per thread at launch (65536 / threads, one CTA per SM) and the
// per-warpgroup split; the sum stays within the launch's total.
constexpr int kRegsSoftmax16 = 192, kRegsIO16 = 120;  // 384 threads, 168 each at launch
// FP8 cache: 80 for the I/O and the widening groups (measured: 72 left the
// I/O code spilling, and 176 / 80 / 80 ran 1-7 % faster than 184 / 72 / 72).
constexpr int kRegsSoftmax8 = 176, kRegsIO8 = 80;     // 512 threads, 128 each at launch
static_assert(128 * kRegsIO16 + 256 * kRegsSoftmax16 <= kThreads16 * 168, "register split exceeds the launch");
static_assert(256 * kRegsIO8 + 256 * kRegsSoftmax8 <= kThreads8 * 128, "register split exceeds the launch");

struct PrefillParams {
    void *out;
    const int32_t *block_tables;
    const int32_t *cu_q;
    const int32_t *seq_lens;
    int max_blocks_per_seq;
    int num_seqs;
    int num_q_heads;
    int group;          // num_q_heads / num_kv_heads
    int heads_per_cta;  // query heads of one kv head that share a tile (<= 16)
    int head_tiles;     // group / heads_per_cta
    int rows_per_head;  // query tokens per tile (multiple of 8)
    int q_pairs;        // ceil(ceil(max_seqlen_q / rows_per_head) / 2)
    int max_q;          // max_seqlen_q: a longer chunk is inconsistent (flagged, not written)
    int num_blocks;
    int block_size;
    int total_q;
    int max_len;        // max_blocks_per_seq * block_size
    int num_kv_heads;
    int num_units;      // q_pairs * num_seqs * num_kv_heads * head_tiles
    int sched_slot;     // this launch's row of g_prefill_sched
    float *part_o;      // stream-K: partial O rows [CTA][slot 2][tile 2][128][D] fp32
    float2 *part_ml;    // stream-K: partial (reference maximum, row sum) [CTA][slot 2][tile 2][128]
    int4 *jobs;         // stream-K: per CTA c, the split unit whose first piece c holds (kNoJob: none):
                        // {last CTA holding a piece, first query row of tile A, query rows from there,
                        //  first query head}
    float scale_log2;   // scale * log2(e) (* k_scale with an FP8 cache)
    float v_scale;      // 1, or the FP8 cache's V scale
};

// One work unit: the two adjacent query tiles A = 2 qp and B = 2 qp + 1 of
// head tile ht of kv head h of sequence s. They share every K/V tile (B's
// queries come later, so B sees at least as many tiles as A). With qp =
// q_pairs - 1 - qr, units are numbered heaviest first, u = ((qr * num_seqs
// + s) * num_kv_heads + h) * head_tiles + ht, when each CTA takes whole
// units from a counter; sequence-major, u = ((s * num_kv_heads + h) *
// head_tiles + ht) * q_pairs + qr, when CTAs take equal shares of the
// tiles (stream-K), so that a sequence's units lie side by side.
struct Unit {
    int s, h, ht, q0, q_len, L;
    int t0[2];       // first query token of tile A / B
    int n[2];        // K/V tiles tile A / B sees (0: the tile has no queries)
};

// What a CTA is handed: K/V tiles j0 <= j < j1 of unit u. CTAs clo..chi
// hold the unit's pieces; clo == chi: the item is the whole unit.
struct Item {
    int u, j0, j1, clo, chi;
};

// Decode unit u; false when tile A has no query rows or the sequence has bad
// offsets or lengths (flagged once, by the unit of the sequence's first
// heads and last query pair, when `flag`).
// A sequence's offsets and length are consistent.
__device__ __forceinline__ bool seq_ok(const PrefillParams &p, int q0, int q_len, int L)
{
    return !(q_len < 0 || q_len > p.max_q || q0 < 0 || q0 + q_len > p.total_q || L < q_len || L > p.max_len);
}

// K/V tiles the unit of query pair qr of a sequence reads (those its tile
// B's last query sees, or tile A's when B has no queries); 0 when tile A
// has no queries.
__device__ __forceinline__ int pair_tiles(const PrefillParams &p, int q_len, int L, int qr)
{
    const int ta = 2 * (p.q_pairs - 1 - qr) * p.rows_per_head;
    if (ta >= q_len)
        return 0;
    return (L - q_len + min(q_len, ta + 2 * p.rows_per_head) + kN - 1) / kN;
}

// SK: the stream-K numbering (sequence-major).
template <bool SK>
__device__ __forceinline__ bool unit_of(const PrefillParams &p, int u, Unit &w, bool flag)
{
    int ht, h, s, qr;
    if constexpr (SK) {
        qr = u % p.q_pairs;
        int r = u / p.q_pairs;
        ht = r % p.head_tiles;
        r /= p.head_tiles;
        h = r % p.num_kv_heads;
        s = r / p.num_kv_heads;
    } else {
        ht = u % p.head_tiles;
        int r = u / p.head_tiles;
        h = r % p.num_kv_heads;
        r /= p.num_kv_heads;
        s = r % p.num_seqs;
        qr = r / p.num_seqs;
    }
    const int q0 = p.cu_q[s], q_len = p.cu_q[s + 1] - q0, L = p.seq_lens[s];
    if (!seq_ok(p, q0, q_len, L)) {
        if (flag && h == 0 && ht == 0 && qr == 0)
            prefill_raise(PA_DEVERR_SEQ_LEN);
        return false;
    }
    const int T = p.rows_per_head;
    const int ta = 2 * (p.q_pairs - 1 - qr) * T;
    if (ta >= q_len)
        return false;
    w.s = s;
    w.h = h;
    w.ht = ht;
    w.q0 = q0;
    w.q_len = q_len;
    w.L = L;
    for (int x = 0; x < 2; ++x) {
        w.t0[x] = ta + x * T;
        const int t_end = min(q_len, w.t0[x] + T);
        w.n[x] = w.t0[x] < q_len ? (L - q_len + t_end + kN - 1) / kN : 0;  // tiles its last query sees
    }
    return true;
}

struct PrefillBars {
    uint64_t q_full, q_empty, k_full[kKStagesMax], k_empty[kKStagesMax], v_full[kVStagesMax], v_empty[kVStagesMax];
    uint64_t q_ready;  // FP8 cache, bf16 queries: the softmax threads have moved Q to fp16
    uint64_t stg_full[2][2];  // FP8 cache: K / V staging half 0 / 1 has landed
    // Per query tile x: s_full[x] its S is in TMEM, p_full[x] its P is,
    // pv_done[x] its O += P V is done (one phase per K/V tile).
    uint64_t s_full[2], p_full[2], pv_done[2];
    uint64_t unit_full[kUnitSlots], unit_empty[kUnitSlots];
    int unit_ring[kUnitSlots];  // unit index, or -1 once the launch's units are all taken
    uint32_t tmem_base;
    int fail;
    // Stream-K: the rest of each work item (first and end K/V tile, first
    // and last CTA holding a piece of the unit; equal: the whole unit).
    int item_ext[kUnitSlots][4];
};

// SPLIT: the stream-K instance (few units, K/V ranges shared out evenly);
// otherwise whole units from a counter.
template <bool BF16, bool FP8, int D, bool SPLIT>
__global__ void __launch_bounds__(threads_for(FP8), 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap kv_map,
                         const __grid_constant__ CUtensorMap q_map, const PrefillParams p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ PrefillBars bars;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = p.rows_per_head, HPC = p.heads_per_cta;
    // Persistent: the Q warp takes the next unit from the launch's counter
    // (skipping units without queries) and hands it to every role through
    // a small ring; the TMA rings and barrier phases run on across units.

    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    auto sQ = [&](int x) { return base + kOffQ + x * kTileBytes; };
    static_assert(D == 64 || D == 128, "head size 64 or 128");
    constexpr int kChunks = D / 64;  // 64-dim, 128-byte-row chunks of a Q/K/V row
    // The MMAs' element type: the query type, except over an FP8 cache, where
    // the codes widen to fp16 in one instruction per pair and bf16 queries
    // are moved to fp16 (kQToF16) by the softmax threads, row by row.
    constexpr bool kMmaBF16 = BF16 && !FP8;
    constexpr bool kQToF16 = BF16 && FP8;
    constexpr int kKStages = FP8 ? kKStages8 : kKStages16;
    constexpr int kVStages = FP8 ? kVStages8 : kVStages16;
    constexpr int kOffV = kOffK + kKStages * kTileBytes;
    constexpr int kOffStage = kOffV + kVStages * kTileBytes;  // FP8: K then V staging tile
    auto sK = [&](int st) { return base + kOffK + st * kTileBytes; };
    auto sV = [&](int st) { return base + kOffV + st * kTileBytes; };
    const uint32_t b_q = smem_addr(&bars.q_full), b_qe = smem_addr(&bars.q_empty);
    const uint32_t b_qr = smem_addr(&bars.q_ready);
    auto b_kf = [&](int st) { return smem_addr(&bars.k_full[st]); };
    auto b_ke = [&](int st) { return smem_addr(&bars.k_empty[st]); };
    auto b_vf = [&](int st) { return smem_addr(&bars.v_full[st]); };
    auto b_ve = [&](int st) { return smem_addr(&bars.v_empty[st]); };
    auto b_s = [&](int x) { return smem_addr(&bars.s_full[x]); };
    auto b_p = [&](int x) { return smem_addr(&bars.p_full[x]); };
    auto b_pv = [&](int x) { return smem_addr(&bars.pv_done[x]); };
    auto b_uf = [&](int i) { return smem_addr(&bars.unit_full[i]); };
    auto b_ue = [&](int i) { return smem_addr(&bars.unit_empty[i]); };

    if (tid == 0) {
        mbar_init(b_q, 1);
        mbar_init(b_qr, 256);  // the 8 softmax warps
        mbar_init(b_qe, 1);
        for (int st = 0; st < kKStages; ++st) {
            mbar_init(b_kf(st), FP8 ? 2 : 1);  // FP8: the two widening warps of the tile
            mbar_init(b_ke(st), 1);
        }
        for (int st = 0; st < kVStages; ++st) {
            mbar_init(b_vf(st), FP8 ? 2 : 1);
            mbar_init(b_ve(st), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(b_s(x), 1);
            mbar_init(b_p(x), 128);
            mbar_init(b_pv(x), 1);
        }
        for (int i = 0; i < 4; ++i)
            mbar_init(smem_addr(&bars.stg_full[i >> 1][i & 1]), 1);
        for (int i = 0; i < kUnitSlots; ++i) {
            mbar_init(b_uf(i), 1);
            mbar_init(b_ue(i), unit_consumers(FP8));
        }
        bars.fail = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&bars.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    auto tS = [&](int x) { return tmem + 128u * x; };        // S of tile x; its P in the first 64 columns
    auto tO = [&](int x) { return tmem + 256u + 128u * x; };  // O of tile x

    // Give up on a wait that runs out (recorded once per CTA); every role then
    // drains to the teardown.
    auto wait_or_fail = [&](uint32_t bar, uint32_t parity) {
        if (mbar_wait(bar, parity))
            return true;
        if (atomicExch(&bars.fail, 1) == 0)
            prefill_raise(PA_DEVERR_TIMEOUT);
        return false;
    };
    // The i-th item handed to this CTA (unit -1: no more). Every lane in
    // `mask` calls it; `leader` arrives once the warp has read the slot.
    // False if the wait ran out.
    auto take_unit = [&](int i, unsigned mask, bool leader, Item &it) {
        const int sl = i % kUnitSlots;
        if (!__all_sync(mask, wait_or_fail(b_uf(sl), (i / kUnitSlots) & 1)))
            return false;
        it.u = *reinterpret_cast<volatile int *>(&bars.unit_ring[sl]);
        if constexpr (SPLIT) {
            const volatile int *e = bars.item_ext[sl];
            it.j0 = e[0];
            it.j1 = e[1];
            it.clo = e[2];
            it.chi = e[3];
        } else {
            it.j0 = 0;
            it.j1 = 0x7fffffff;
            it.clo = it.chi = 0;
        }
        __syncwarp(mask);
        if (leader)
            mbar_arrive(b_ue(sl));
        return true;
    };

    // Register split, per warpgroup (each of its four warps runs the same
    // instruction): the K/V/MMA/Q group (and with an FP8 cache the widening
    // group) drops to kRegsIO16 / kRegsIO8, the two softmax groups rise to
    // kRegsSoftmax16 / kRegsSoftmax8; the sum stays within the launch's total.
    if (warp >= 8) {
    if constexpr (FP8)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIO8));
    else
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIO16));
    if (warp == kWarpQ) {
        // ------------------------------------------------------------ Q
        // Scheduler and Q: find this CTA's next work item, hand it on, and
        // load its two query tiles once the previous item's last S = Q K^T
        // has completed. Whole units come from the launch's counter; under
        // stream-K, CTA c takes tiles [c W / G, (c + 1) W / G) of the W K/V
        // tiles of all units laid end to end (G CTAs), cut at unit ends.
        const int H = p.num_kv_heads * p.head_tiles;  // units of one query pair of a sequence
        auto seq_tiles = [&](int s, bool flag) {     // K/V tiles of one head tile of sequence s
            const int q0 = p.cu_q[s], q_len = p.cu_q[s + 1] - q0, L = p.seq_lens[s];
            if (!seq_ok(p, q0, q_len, L)) {
                if (flag)
                    prefill_raise(PA_DEVERR_SEQ_LEN);
                return 0LL;
            }
            long long a = 0;
            for (int qr = 0; qr < p.q_pairs; ++qr)
                a += pair_tiles(p, q_len, L, qr);
            return a;
        };
        long long lo = 0, hi = 0, W = 0, Ts = 0;  // this CTA's tiles [lo, hi); sequence ws starts at tile Ts
        long long G = 1;                           // CTAs sharing the tiles: at most one per tile, so that
        int ws = 0;                                // every share is non-empty
        if constexpr (SPLIT) {
            long long part = 0;
            for (int s = lane; s < p.num_seqs; s += 32)
                part += H * seq_tiles(s, true);
            for (int o = 16; o > 0; o >>= 1)
                part += __shfl_xor_sync(kFull, part, o);
            W = part;
            G = min((long long)gridDim.x, max(W, 1LL));
            if (blockIdx.x < G) {
                lo = (long long)blockIdx.x * W / G;
                hi = ((long long)blockIdx.x + 1) * W / G;
            }
            long long done = 0;  // tiles of the sequences before this group of 32
            for (int s0 = 0; lo < hi && s0 < p.num_seqs; s0 += 32) {
                const int s = s0 + lane;
                const long long wq = s < p.num_seqs ? H * seq_tiles(s, false) : 0;
                long long incl = wq;
                for (int o = 1; o < 32; o <<= 1) {
                    const long long v = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o)
                        incl += v;
                }
                const long long start = done + incl - wq;
                const unsigned hit = __ballot_sync(kFull, wq > 0 && start <= lo && lo < start + wq);
                if (hit) {
                    const int src = __ffs(hit) - 1;
                    ws = s0 + src;
                    Ts = __shfl_sync(kFull, start, src);
                    break;
                }
                done += __shfl_sync(kFull, incl, 31);
            }
        }
        if (lane == 0) {
            int* next = &g_prefill_sched[p.sched_slot][0];
            // Stream-K walk: unit (ws, hh, qr) holds tiles [Tu, Tu + nu).
            int hh = 0, qr = 0, wq_len = 0, wL = 0, nu = 0;
            bool wok = false;
            long long Tu = 0, pos = lo;
            auto enter_seq = [&]() {
                const int q0 = p.cu_q[ws];
                wq_len = p.cu_q[ws + 1] - q0;
                wL = p.seq_lens[ws];
                wok = seq_ok(p, q0, wq_len, wL);
            };
            auto tiles_here = [&]() { return wok ? pair_tiles(p, wq_len, wL, qr) : 0; };
            if (SPLIT && lo < hi) {
                enter_seq();
                const long long a = seq_tiles(ws, false);
                hh = a > 0 ? (int)((lo - Ts) / a) : 0;
                Tu = Ts + hh * a;
                nu = tiles_here();
                while (Tu + nu <= lo && qr + 1 < p.q_pairs) {
                    Tu += nu;
                    ++qr;
                    nu = tiles_here();
                }
            }
            auto cta_of = [&](long long t) { return (int)(((t + 1) * G - 1) / W); };
            if constexpr (SPLIT)
                p.jobs[blockIdx.x] = make_int4(-1, 0, 0, 0);
            for (int i = 0;; ++i) {
                Unit w;
                Item it = {-1, 0, 0, 0, 0};
                if constexpr (SPLIT) {
                    if (pos < hi && nu > 0 && Tu <= pos && pos < Tu + nu) {
                        it.u = ((ws * H) + hh) * p.q_pairs + qr;
                        const long long end = min(Tu + nu, hi);
                        it.j0 = (int)(pos - Tu);
                        it.j1 = (int)(end - Tu);
                        it.clo = cta_of(Tu);
                        it.chi = cta_of(Tu + nu - 1);
                        pos = end;
                        // On to the next unit with tiles (bounded: every step
                        // moves (ws, hh, qr) forward).
                        while (pos < hi) {
                            Tu += nu;
                            nu = 0;
                            if (++qr == p.q_pairs) {
                                qr = 0;
                                if (++hh == H) {
                                    hh = 0;
                                    if (++ws >= p.num_seqs)
                                        break;
                                    enter_seq();
                                }
                            }
                            nu = tiles_here();
                            if (nu > 0)
                                break;
                        }
                        if (!unit_of<true>(p, it.u, w, false))
                            it.u = -1;
                        else if (it.j0 == 0 && it.chi > it.clo)  // this CTA holds the unit's first piece
                            p.jobs[blockIdx.x] = make_int4(it.chi, w.q0 + w.t0[0], w.q_len - w.t0[0],
                                                           w.h * p.group + w.ht * HPC);
                    }
                } else {
                    int u;
                    do {
                        u = atomicAdd(next, 1);
                    } while (u < p.num_units && !unit_of<false>(p, u, w, true));
                    if (u < p.num_units) {
                        it.u = u;
                        it.j1 = 0x7fffffff;
                    }
                }
                const int sl = i % kUnitSlots;
                if (i >= kUnitSlots && !wait_or_fail(b_ue(sl), ((i / kUnitSlots) - 1) & 1))
                    break;
                bars.unit_ring[sl] = it.u;
                if constexpr (SPLIT) {
                    bars.item_ext[sl][0] = it.j0;
                    bars.item_ext[sl][1] = it.j1;
                    bars.item_ext[sl][2] = it.clo;
                    bars.item_ext[sl][3] = it.chi;
                }
                mbar_arrive(b_uf(sl));
                if (it.u < 0)
                    break;
                if (i > 0 && !wait_or_fail(b_qe, (i - 1) & 1))
                    break;
                const int head0 = w.h * p.group + w.ht * HPC;
                const int tiles = w.n[1] > 0 ? 2 : 1;
                mbar_expect_tx(b_q, (uint32_t)(tiles * kChunks * HPC * T * 128));
                for (int x = 0; x < tiles; ++x)
                    for (int c = 0; c < kChunks; ++c)
                        for (int g = 0; g < HPC; ++g)
                            tma_load_3d(sQ(x) + c * kChunkBytes + g * T * 128, &q_map, b_q, c * 64, head0 + g,
                                        w.q0 + w.t0[x]);
            }
        }
    } else if (warp == kWarpK || warp == kWarpV) {
        // ---------------------------------------------------------- K, V
        const bool is_k = warp == kWarpK;
        if constexpr (!FP8) {
            // Warp 8 produces the K tiles, warp 10 the V tiles, each at its own
            // pace through its ring; lane i < 8 moves the 16-token box i of each
            // tile. The block-table entry of the next tile is loaded while the
            // current one waits for its stage.
            if (lane < 8) {
                const int box = lane, leader = 0;
                const unsigned group_mask = 0x000000FFu;
                const int stages = is_k ? kKStages : kVStages;
                int gc = 0;  // K (or V) tiles produced by this CTA so far
                bool go = true;
                for (int i = 0; go; ++i) {
                    Item it;
                    if (!take_unit(i, group_mask, lane == leader, it) || it.u < 0)
                        break;
                    Unit w;
                    unit_of<SPLIT>(p, it.u, w, false);
                    const int n = SPLIT ? min(max(w.n[0], w.n[1]), it.j1) : max(w.n[0], w.n[1]);
                    const int32_t *table = p.block_tables + (long long)w.s * p.max_blocks_per_seq;
                    auto lookup = [&](int j) {
                        const int kt = j * kN + kBoxTokens * box;
                        return (j < n && kt < w.L) ? __ldg(table + kt / p.block_size) : -1;
                    };
                    int next = lookup(it.j0);
                    for (int j = it.j0; j < n; ++j, ++gc) {
                        int phys = next;
                        next = lookup(j + 1);
                        const int st = gc % stages;
                        if (gc >= stages &&
                            !wait_or_fail(is_k ? b_ke(st) : b_ve(st), ((gc - stages) / stages) & 1)) {
                            go = false;
                            break;
                        }
                        const int kt = j * kN + kBoxTokens * box;
                        const int tib = kt % p.block_size;
                        if (phys >= p.num_blocks || (phys < 0 && kt < w.L)) {
                            prefill_raise(PA_DEVERR_BLOCK_ID);
                            phys = p.num_blocks;
                        }
                        if (phys < 0)
                            phys = p.num_blocks;  // past the sequence end: outside the map, zeros
                        const uint32_t full = is_k ? b_kf(st) : b_vf(st);
                        if (lane == leader)
                            mbar_expect_tx(full, kChunks * kChunkBytes);
                        __syncwarp(group_mask);
                        const uint32_t dst = (is_k ? sK(st) : sV(st)) + box * (kBoxTokens * 128);
                        for (int c = 0; c < kChunks; ++c)
                            tma_load_5d(dst + c * kChunkBytes, &kv_map, full, c * 64, w.h, tib, phys, is_k ? 0 : 1);
                    }
                }
            }
        }
    } else if (FP8 && warp >= 12) {
        // ------------------------------------------------- FP8 widening
        // Warps 12-15: K rows 0-63, K rows 64-127, V rows 0-63, V rows
        // 64-127 of every tile. Lanes 0-3 bring the half tile's four 16-token
        // boxes of codes into this warp's staging buffer (TMA; 128-byte rows
        // with the 128-byte swizzle at head size 128, plain 64-byte rows at
        // 64); the whole warp widens them, exactly, into the 16-bit ring
        // stage in the MMA's layout (rows past the sequence end as zeros),
        // arrives on the stage's full barrier (two arrivals make it full)
        // and requests its half of the next tile.
        const int cw = warp - 12, part = cw & 1;
        const bool is_k = cw < 2;
        const uint32_t stg = base + kOffStage + cw * (kStageBytes8 / 2);
        const uint32_t b_stg = smem_addr(&bars.stg_full[cw >> 1][part]);
        const int stages = is_k ? kKStages : kVStages;
        int gc = 0;  // tiles produced by this CTA so far
        bool go = true;
        for (int i = 0; go; ++i) {
            Item it;
            if (!take_unit(i, kFull, lane == 0, it) || it.u < 0)
                break;
            Unit w;
            unit_of<SPLIT>(p, it.u, w, false);
            const int n = SPLIT ? min(max(w.n[0], w.n[1]), it.j1) : max(w.n[0], w.n[1]);
            const int32_t *table = p.block_tables + (long long)w.s * p.max_blocks_per_seq;
            auto issue = [&](int j) {
                if (lane < 4) {
                    const int kt = j * kN + part * (kN / 2) + kBoxTokens * lane;
                    int phys = kt < w.L ? __ldg(table + kt / p.block_size) : -1;
                    if (phys >= p.num_blocks || (phys < 0 && kt < w.L)) {
                        prefill_raise(PA_DEVERR_BLOCK_ID);
                        phys = p.num_blocks;
                    }
                    if (phys < 0)
                        phys = p.num_blocks;  // past the sequence end: outside the map, zeros
                    if (lane == 0)
                        mbar_expect_tx(b_stg, (kN / 2) * D);
                    __syncwarp(0xFu);
                    tma_load_5d(stg + lane * (kBoxTokens * D), &kv_map, b_stg, 0, w.h, kt % p.block_size, phys,
                                is_k ? 0 : 1);
                }
            };
            issue(it.j0);
            for (int j = it.j0; j < n; ++j, ++gc) {
                const int st = gc % stages;
                if (!__all_sync(kFull, wait_or_fail(b_stg, gc & 1)) ||
                    (gc >= stages && !__all_sync(kFull, wait_or_fail(is_k ? b_ke(st) : b_ve(st),
                                                                     ((gc - stages) / stages) & 1)))) {
                    go = false;
                    break;
                }
                const uint32_t dst = is_k ? sK(st) : sV(st);
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int rh = lane + 32 * rr;          // row within the half
                    const int r = part * (kN / 2) + rh;    // row within the tile
                    const bool pad = j * kN + r >= w.L;
#pragma unroll
                    for (int qi = 0; qi < D / 16; ++qi) {
                        // The 16-byte unit q of codes (dims 16q .. 16q + 15).
                        // At head size 64 the rows are 64 bytes, unswizzled:
                        // lane pairs take the units in the order q = qi ^ h(a),
                        // a = (row / 2) % 4, h = multiplication by a generator
                        // of GF(4) (0, 2, 3, 1), so that both h(a) and
                        // h(a) ^ a run over all four units and neither these
                        // loads nor the swizzled stores below meet a bank
                        // conflict within a quarter warp.
                        const int q = D == 128 ? qi : qi ^ ((0x78 >> (2 * ((rh >> 1) & 3))) & 3);
                        const uint32_t src = D == 128 ? stg + rh * 128 + ((q ^ (rh & 7)) << 4) : stg + rh * 64 + (q << 4);
                        const uint4 c = pad ? make_uint4(0u, 0u, 0u, 0u) : lds128(src);
                        // fp16 whatever the query type: the MMAs of the FP8
                        // path run in fp16 (bf16 queries are moved to fp16).
                        const uint32_t h[8] = {e4m3_pair_lo(c.x), e4m3_pair_hi(c.x), e4m3_pair_lo(c.y),
                                               e4m3_pair_hi(c.y), e4m3_pair_lo(c.z), e4m3_pair_hi(c.z),
                                               e4m3_pair_lo(c.w), e4m3_pair_hi(c.w)};
                        // dims 16q .. 16q + 15: chunk q / 4, 16-byte units 2 (q % 4) and + 1
                        const uint32_t row = dst + (q >> 2) * kChunkBytes + r * 128;
                        const int u0 = 2 * (q & 3);
                        sts128(row + ((u0 ^ (r & 7)) << 4), h[0], h[1], h[2], h[3]);
                        sts128(row + (((u0 + 1) ^ (r & 7)) << 4), h[4], h[5], h[6], h[7]);
                    }
                }
                fence_proxy_async();  // widened rows for the MMA; staging reads before its reuse
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(is_k ? b_kf(st) : b_vf(st));
                if (j + 1 < n)
                    issue(j + 1);
            }
        }
    } else if (warp == kWarpMMA) {
        // ---------------------------------------------------------- MMA
        // Per K/V tile j: S_A(0), S_B(0) up front, then for each tile x in
        // turn O_x += P_x V_j followed by S_x(j + 1) = Q_x K_{j+1}^T, so the
        // scores of one tile are computed while the other tile's softmax
        // runs. S_x(j + 1) overwrites P_x(j) in TMEM: MMAs complete in issue
        // order, so the P V that reads it is done first.
        if (lane == 0) {
            const uint32_t id_s = instr_desc(kM, kN, kMmaBF16, false);
            const uint32_t id_o = instr_desc(kM, D, kMmaBF16, true);
            // Descriptors are built once per operand tile; each k step adds
            // its byte offset / 16 to the start-address field (bits 0-13,
            // which cannot carry: shared memory ends below 256 KB).
            auto issue_s = [&](int x, int ks) {
                const uint64_t dq = smem_desc(sQ(x), 16, 1024), dk = smem_desc(sK(ks), 16, 1024);
                const uint32_t ts = tS(x);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t off = (uint64_t)(((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4);
                    tc_mma(ts, dq + off, dk + off, id_s, k > 0 ? 1u : 0u);
                }
                tc_commit(b_s(x));
            };
            int kc = 0, vc = 0, ui = 0;  // K tiles, V tiles and units consumed so far
            int gx[2] = {0, 0};          // P V of tile x issued so far
            bool go = true;
            for (int i = 0; go; ++i) {
                Item it;
                if (!take_unit(i, 1u, true, it) || it.u < 0)
                    break;
                Unit w;
                unit_of<SPLIT>(p, it.u, w, false);
                // Tiles j0 <= j < j1 of the unit; tile x reads those below its ne[x].
                const int j0 = SPLIT ? it.j0 : 0;
                const int j1 = SPLIT ? min(max(w.n[0], w.n[1]), it.j1) : max(w.n[0], w.n[1]);
                const int ne_piece[2] = {min(w.n[0], j1), min(w.n[1], j1)};
                const int *ne = SPLIT ? ne_piece : w.n;
                if (!wait_or_fail(kQToF16 ? b_qr : b_q, ui & 1))
                    break;
                ++ui;
                tc_fence_after();
                {
                    const int ks = kc % kKStages;
                    if (!wait_or_fail(b_kf(ks), (kc / kKStages) & 1))
                        break;
                    tc_fence_after();
                    for (int x = 0; x < 2; ++x)
                        if (ne[x] > j0)
                            issue_s(x, ks);
                    tc_commit(b_ke(ks));
                    ++kc;
                    if (j1 - j0 == 1)
                        tc_commit(b_qe);  // Q free once the item's last scores are done
                }
                for (int j = j0; go && j < j1; ++j) {
                    const int vs = vc % kVStages;
                    if (!wait_or_fail(b_vf(vs), (vc / kVStages) & 1)) {
                        go = false;
                        break;
                    }
                    int ks_next = -1;
                    for (int x = 0; x < 2; ++x) {
                        if (j >= ne[x])
                            continue;
                        if (!wait_or_fail(b_p(x), gx[x] & 1)) {
                            go = false;
                            break;
                        }
                        tc_fence_after();
                        // O_x += P_x V: A = P from TMEM (8 columns per 16
                        // tokens), B = V (MN-major: 64-dim chunks 16 KB apart,
                        // 8-token groups 1 KB apart).
                        const uint64_t dv = smem_desc(sV(vs), kChunkBytes, 1024);
                        const uint32_t to = tO(x), ts = tS(x);
#pragma unroll
                        for (int k = 0; k < kN / 16; ++k)
                            tc_mma_ts(to, ts + k * 8, dv + (uint64_t)(k * (2048 >> 4)), id_o,
                                      (j > j0 || k > 0) ? 1u : 0u);
                        tc_commit(b_pv(x));
                        ++gx[x];
                        // The tile's last O += P V is issued: V's stage is
                        // free once it completes (tile B, if it reads V_j,
                        // comes after tile A).
                        if (x == 1 || j >= ne[1])
                            tc_commit(b_ve(vs));
                        if (j + 1 < ne[x]) {
                            if (ks_next < 0) {
                                ks_next = kc % kKStages;
                                if (!wait_or_fail(b_kf(ks_next), (kc / kKStages) & 1)) {
                                    go = false;
                                    break;
                                }
                                tc_fence_after();
                            }
                            issue_s(x, ks_next);
                        }
                    }
                    if (!go)
                        break;
                    if (ks_next >= 0) {
                        tc_commit(b_ke(ks_next));
                        ++kc;
                        if (j + 2 == j1)
                            tc_commit(b_qe);
                    }
                    ++vc;
                }
            }
        }
        __syncwarp();
    }
    } else {
    if constexpr (FP8)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax8));
    else
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax16));
    {
        // ---------------------------------------------------- softmax rows
        // Warpgroup x (warps 4x .. 4x + 3) owns query tile x; each thread one
        // row (TMEM lane). Per K/V tile: read S, mask it causally, run the
        // fp32 online softmax in base 2 (the reference maximum moves only
        // when a score exceeds it by 2^8, so O in TMEM is rarely rescaled),
        // and write P, rounded to the element type, over the row's first 64
        // S columns for the P V MMA. At the end of the unit, divide O by the
        // row sum and store.
        const int x = warp >> 2, quarter = warp & 3;
        const int r = quarter * 32 + lane;  // this thread's TMEM lane (row)
        const int g = r / T, t = r - g * T;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        float sc = p.scale_log2;  // this row's score factor (base 2)
        const bool sc_pos = sc >= 0.f;
        int gx = 0, vbase = 0;  // tiles of this query tile, and V tiles of the CTA, so far
        bool alive = true;
        for (int i = 0; alive; ++i) {
            Item it;
            if (!take_unit(i, kFull, lane == 0, it) || it.u < 0)
                break;
            Unit w;
            unit_of<SPLIT>(p, it.u, w, false);
            // This tile reads K/V tiles j0 <= j < nx of the item's j0 .. j1.
            const int j0 = SPLIT ? it.j0 : 0;
            const int j1 = SPLIT ? min(max(w.n[0], w.n[1]), it.j1) : max(w.n[0], w.n[1]);
            const int nx = SPLIT ? min(w.n[x], j1) : w.n[x];
            // The K/V tile holding the sequence end (padding slots past it)
            // is zeroed in V by the first tile that reads it.
            const int jp = (w.L % kN) ? w.L / kN : -1;
            const bool zeroes = !FP8 && jp >= j0 && jp < nx && (x == 0 || jp >= (SPLIT ? min(w.n[0], j1) : w.n[0]));
            const bool valid = g < HPC && w.t0[x] + t < w.q_len;
            const int pos = valid ? w.L - w.q_len + w.t0[x] + t : -1;  // last token this row sees
            if constexpr (kQToF16) {
                // Move Q row r of this tile to fp16 in place, scaled by 2^-e
                // so that the row's largest magnitude lies in [2^14, 2^15):
                // exact for every element within 2^31 of that maximum, and
                // no overflow. This thread also owns score row r, so 2^e
                // joins its score factor. A row holding Inf or NaN keeps
                // e = 0 (and yields NaN, as the definition does).
                if (!__all_sync(kFull, wait_or_fail(b_q, i & 1))) {
                    alive = false;
                    break;
                }
                sc = p.scale_log2;
                if (nx > j0) {
                    const uint32_t row = sQ(x) + r * 128;
                    uint4 qv[kChunks * 8];
                    uint32_t mag = 0;  // largest |q| as bf16 bits, per half
#pragma unroll
                    for (int k = 0; k < kChunks * 8; ++k) {
                        qv[k] = lds128(row + (k >> 3) * kChunkBytes + (((k & 7) ^ (r & 7)) << 4));
                        mag = __vmaxu2(mag, __vmaxu2(qv[k].x & 0x7FFF7FFFu, qv[k].y & 0x7FFF7FFFu));
                        mag = __vmaxu2(mag, __vmaxu2(qv[k].z & 0x7FFF7FFFu, qv[k].w & 0x7FFF7FFFu));
                    }
                    mag = max(mag & 0xFFFFu, mag >> 16);
                    const int field = (int)(mag >> 7);  // biased exponent (0: zero or subnormal)
                    const int e = field == 255 ? 0 : field == 0 ? (mag ? -120 : 0) : max(field - 141, -120);
                    const float down = __int_as_float((127 - e) << 23);  // 2^-e
                    sc = p.scale_log2 * __int_as_float((127 + e) << 23);
                    auto to_f16 = [&](uint32_t b) {
                        const __half2 h = __floats2half2_rn(__uint_as_float(b << 16) * down,
                                                            __uint_as_float(b & 0xFFFF0000u) * down);
                        return *reinterpret_cast<const uint32_t *>(&h);
                    };
#pragma unroll
                    for (int k = 0; k < kChunks * 8; ++k)
                        sts128(row + (k >> 3) * kChunkBytes + (((k & 7) ^ (r & 7)) << 4), to_f16(qv[k].x),
                               to_f16(qv[k].y), to_f16(qv[k].z), to_f16(qv[k].w));
                }
                fence_proxy_async();  // the fp16 rows, for the score MMAs
                mbar_arrive(b_qr);
            }
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = j0; j < nx; ++j, ++gx) {
                if (!__all_sync(kFull, wait_or_fail(b_s(x), gx & 1))) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                float sv[kN];
                {
                    const uint32_t ta = tS(x) + lane_off;
                    uint32_t *rv = reinterpret_cast<uint32_t *>(sv);
#pragma unroll
                    for (int c = 0; c < kN / 32; ++c)
                        tc_ld32_async(ta + c * 32, rv + c * 32);
                    tc_wait_ld();
                }
                const int kb = j * kN;
                // Causal mask: a score this row must not see becomes -inf
                // (+inf for a negative scale): neutral for the extremum
                // below, and its weight 2^(s scale - ref) is exactly 0, so
                // the tile then runs the same branch-free code as a full one.
                // Padding slots past the sequence end (whatever they hold,
                // NaN included) are masked the same way.
                if (kb + kN - 1 > pos) {
                    const float masked = sc_pos ? -INFINITY : INFINITY;
#pragma unroll
                    for (int c = 0; c < kN; ++c)
                        sv[c] = kb + c <= pos ? sv[c] : masked;
                }
                // Row maximum in base 2: scale x the largest visible raw score
                // (the smallest for a negative scale; rounding is monotone, so
                // this is the largest scaled score exactly); 8 chains.
                float e8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    e8[i] = sc_pos ? -INFINITY : INFINITY;
                if (sc_pos) {
#pragma unroll
                    for (int c = 0; c < kN; c += 2)
                        e8[(c >> 1) & 7] = max3(e8[(c >> 1) & 7], sv[c], sv[c + 1]);
                } else {
#pragma unroll
                    for (int c = 0; c < kN; c += 2)
                        e8[(c >> 1) & 7] = min3(e8[(c >> 1) & 7], sv[c], sv[c + 1]);
                }
                const float e = sc_pos ? fmaxf(fmaxf(fmaxf(e8[0], e8[1]), fmaxf(e8[2], e8[3])),
                                               fmaxf(fmaxf(e8[4], e8[5]), fmaxf(e8[6], e8[7])))
                                       : fminf(fminf(fminf(e8[0], e8[1]), fminf(e8[2], e8[3])),
                                               fminf(fminf(e8[4], e8[5]), fminf(e8[6], e8[7])));
                const float mx = (e == INFINITY || e == -INFINITY) ? -INFINITY : __fmul_rn(e, sc);
                // The reference maximum moves only when a score exceeds it by
                // more than kRescaleLog2 (P then stays <= 2^kRescaleLog2, which
                // the element type holds with full relative precision).
                const bool grow = mx > m_run + kRescaleLog2;
                const float m_new = grow ? mx : m_run;
                const float alpha = grow ? ex2(m_run - m_new) : 1.f;
                const float ref = m_new == -INFINITY ? 0.f : m_new;
                // P = 2^(s scale - ref), rounded to the element type, packed in
                // pairs (the lower-indexed token in the low half); the row sum
                // adds the same rounded values. The argument is one fused
                // multiply-add while |ref| < 2^20: its residual against the
                // rounded maximum is then below 2^-4, so P <= 2^8.1. A warp
                // holding a larger reference rounds each product before the
                // subtraction, as for the maximum, so that the largest
                // score's argument is exactly mx - ref <= 2^8 however large
                // the scores (a fused residual can reach half an ulp of them).
                uint32_t pw[kN / 2];
                float l8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    l8[i] = 0.f;
                auto fill = [&](auto fused) {
                    auto p_of = [&](float s) {
                        if constexpr (decltype(fused)::value)
                            return ex2(fmaf(s, sc, -ref));
                        else
                            return ex2(__fmul_rn(s, sc) - ref);
                    };
                    if constexpr (decltype(fused)::value) {
                        // Two columns per step: the argument by one packed
                        // fused multiply-add (the same value as fmaf), then
                        // 2^x from the MUFU unit (or, every kPolyEvery-th
                        // pair if enabled, from the FMA-pipe polynomial).
                        const uint64_t sc2 = pk2(sc, sc), nref2 = pk2(-ref, -ref);
#pragma unroll
                        for (int c = 0; c < kN / 2; ++c) {
                            const uint64_t x2 = fma2(pk2(sv[2 * c], sv[2 * c + 1]), sc2, nref2);
                            float p0, p1;
                            if (kPolyEvery > 0 && c % (kPolyEvery > 0 ? kPolyEvery : 1) == kPolyEvery - 1) {
                                exp2_poly2<kMmaBF16 ? 3 : 4>(x2, p0, p1);
                            } else {
                                float x0, x1;
                                unpk2(x2, x0, x1);
                                p0 = ex2(x0);
                                p1 = ex2(x1);
                            }
                            pw[c] = pack2<kMmaBF16>(p0, p1);
                            l8[c & 7] = add_pair<kMmaBF16>(l8[c & 7], pw[c]);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < kN / 2; ++c) {
                            pw[c] = pack2<kMmaBF16>(p_of(sv[2 * c]), p_of(sv[2 * c + 1]));
                            l8[c & 7] = add_pair<kMmaBF16>(l8[c & 7], pw[c]);
                        }
                    }
                };
                if (__all_sync(kFull, fabsf(ref) < 0x1p20f))
                    fill(std::true_type{});
                else
                    fill(std::false_type{});
                if (sc == 0.f && kb + kN - 1 > pos) {
                    // Scale 0: a masked score would have given 0 x inf = NaN.
                    // Every visible token weighs 2^-ref, every masked one 0.
                    const float pv = ex2(-ref);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        l8[i] = 0.f;
#pragma unroll
                    for (int c = 0; c < kN / 2; ++c) {
                        pw[c] = pack2<kMmaBF16>(kb + 2 * c <= pos ? pv : 0.f, kb + 2 * c + 1 <= pos ? pv : 0.f);
                        l8[c & 7] = add_pair<kMmaBF16>(l8[c & 7], pw[c]);
                    }
                }
                const float ls = ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
                // Rescale O when the reference moved. The previous tile's
                // O += P V is done: it was issued before this tile's S, whose
                // completion was awaited above.
                if (j > j0 && __any_sync(kFull, alpha != 1.f)) {
                    const uint32_t to = tO(x) + lane_off;
                    float o[32];
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        tc_ld32(to + c * 32, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] *= alpha;
                        tc_st32(to + c * 32, o);
                    }
                }
                // P over the row's first 64 S columns (already read).
                tc_st32u(tS(x) + lane_off, pw);
                tc_st32u(tS(x) + lane_off + 32, pw + 32);
                l_run = l_run * alpha + ls;
                m_run = m_new;
                // The V rows past the sequence end hold whatever the pool's
                // padding slots hold: zero them (P is 0 there) once V lands.
                if (zeroes && j == jp) {
                    const int vt = vbase + (j - j0), vs = vt % kVStages;
                    if (!__all_sync(kFull, wait_or_fail(b_vf(vs), (vt / kVStages) & 1))) {
                        alive = false;
                        break;
                    }
                    if (kb + r >= w.L)
                        for (int c = 0; c < kChunks; ++c)
                            for (int i = 0; i < 8; ++i)
                                sts128(sV(vs) + c * kChunkBytes + r * 128 + i * 16, 0u, 0u, 0u, 0u);
                    fence_proxy_async();
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                mbar_arrive(b_p(x));
            }
            if (!alive)
                break;
            vbase += j1 - j0;
            const bool whole = !SPLIT || it.clo == it.chi, work = nx > j0;
            if (w.n[x] == 0 || (whole && !work))
                continue;  // the tile has no queries (or, whole, no tiles)
            // Item epilogue. Reading O here comes before this row's first P
            // of the next item, and so before its first P V overwrites O.
            if (work) {
                if (!__all_sync(kFull, wait_or_fail(b_pv(x), (gx - 1) & 1))) {
                    alive = false;
                    break;
                }
                tc_fence_after();
            }
            uint16_t *out = static_cast<uint16_t *>(p.out) +
                            ((long long)(w.q0 + w.t0[x] + t) * p.num_q_heads + w.h * p.group + w.ht * HPC + g) * D;
            const uint32_t to = tO(x) + lane_off;
            float o[32];
            auto store_row = [&](int c, const float *v, float inv) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 e;
                    e.x = pack2<BF16>(v[8 * q + 0] * inv, v[8 * q + 1] * inv);
                    e.y = pack2<BF16>(v[8 * q + 2] * inv, v[8 * q + 3] * inv);
                    e.z = pack2<BF16>(v[8 * q + 4] * inv, v[8 * q + 5] * inv);
                    e.w = pack2<BF16>(v[8 * q + 6] * inv, v[8 * q + 7] * inv);
                    reinterpret_cast<uint4 *>(out + c * 32)[q] = e;
                }
            };
            if (whole) {
                // O / l for the valid rows.
                const float inv = l_run > 0.f ? p.v_scale / l_run : 0.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    tc_ld32(to + c * 32, o);
                    if (valid)
                        store_row(c, o, inv);
                }
                continue;
            }
            // A piece of a split unit: store this piece's partial softmax
            // state for paged_prefill_merge_kernel (O relative to 2^m, the
            // reference maximum m, the row sum l; a tile with no K/V tile in
            // the piece stores the empty state m = -inf, l = 0, O = 0).
            // Slot: CTA c holds at most two partial pieces, the unit it
            // starts inside (slot 0) and the one it starts and leaves
            // unfinished (slot 1).
            {
                const int slot = (((int)blockIdx.x * 2 + ((int)blockIdx.x == it.clo ? 1 : 0)) * 2 + x) * kM + r;
                float4 *po = reinterpret_cast<float4 *>(p.part_o + (size_t)slot * D);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    if (work) {
                        tc_ld32(to + c * 32, o);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = 0.f;
                    }
                    if (valid)
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            po[c * 8 + q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                }
                if (valid)
                    p.part_ml[slot] = work ? make_float2(m_run, l_run) : make_float2(-INFINITY, 0.f);
            }
        }
    }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Every role has left its loop, so this CTA takes no more units; the
    // last CTA to get here resets the launch's counters for the next use
    // (a stream-K launch uses none).
    if (!SPLIT && tid == 0) {
        __threadfence();
        if (atomicAdd(&g_prefill_sched[p.sched_slot][1], 1) == (int)gridDim.x - 1) {
            g_prefill_sched[p.sched_slot][0] = 0;
            g_prefill_sched[p.sched_slot][1] = 0;
            __threadfence();
        }
    }
    if (warp == kWarpMMA)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
}

// Stream-K merge ([book] §4.6: partial softmax states over disjoint token
// ranges combine exactly). For each split unit (the job record of the CTA
// holding its first piece) and each valid row of its tiles, the pieces'
// states (m_c, l_c, O_c) are folded with the online rule (M the running
// maximum, earlier terms rescaled by 2^(M_old - M_new)); out = O / L. A
// thread takes 4 columns of a row. With Q > 1 "planes", plane q folds the
// pieces c0 + q, c0 + q + Q, ... in order and the Q partial states are
// then combined in plane order through shared memory, so that a unit cut
// into many pieces is merged by many threads; with Q = 1 a thread folds all
// pieces of kMergeRowsPerThread rows (their loads in flight together).
// Either way the order is fixed, so the result does not depend on which
// piece finished first. Blocks go to the jobs in CTA order (block b: the
// b / (2 * blocks per tile)-th job), found by one warp's scan of the job
// records. Waits for the main kernel (programmatic dependent launch).
template <int D, int Q>
struct MergeGeo {
    static constexpr int kTpr = D / 4;                      // threads per row (4 columns each)
    static constexpr int kRows = 256 / (kTpr * Q);          // rows per pass of the block
    static constexpr int kRpt = Q == 1 ? kMergeRowsPerThread : 1;
    static constexpr int kBlockRows = kRows * kRpt;
    static constexpr int kBlocks = kM / kBlockRows;         // blocks per 128-row tile
};

template <bool BF16, int D, int Q>
__global__ void __launch_bounds__(256) paged_prefill_merge_kernel(const PrefillParams p, int grid_main)
{
    using Geo = MergeGeo<D, Q>;
    constexpr int kTpr = Geo::kTpr, kRows = Geo::kRows, kRpt = Geo::kRpt;
    const int job_k = blockIdx.x / (2 * Geo::kBlocks), x = (blockIdx.x / Geo::kBlocks) & 1,
              rb = blockIdx.x % Geo::kBlocks;
    const int tid = threadIdx.x, lane = tid & 31;
    const int tpr = tid % kTpr, q = (tid / kTpr) % Q, rsub = tid / (kTpr * Q);
    __shared__ int s_c;
    __shared__ float s_st[Q > 1 ? kRows * Q * kTpr * 6 : 1];
    grid_dependency_wait();
    if (tid < 32) {
        int found = -1, seen = 0;
        for (int c0 = 0; c0 < grid_main && found < 0; c0 += 32) {
            const int c = c0 + lane;
            bool v = false;
            if (c < grid_main) {
                const int last = p.jobs[c].x;
                v = last > c && last < grid_main;
            }
            unsigned m = __ballot_sync(0xFFFFFFFFu, v);
            const int cnt = __popc(m);
            if (job_k < seen + cnt) {
                for (int t = job_k - seen; t > 0; --t)
                    m &= m - 1;
                found = c0 + __ffs(m) - 1;
            }
            seen += cnt;
        }
        if (lane == 0)
            s_c = found;
    }
    __syncthreads();
    const int c = s_c;
    if (c < 0)
        return;
    const int4 job = p.jobs[c];  // {last CTA, first row of tile A, rows from there, first head}
    const int T = p.rows_per_head;
    float M[kRpt], L[kRpt], A[kRpt][4];
    int slot0[kRpt];
    bool ok[kRpt];
#pragma unroll
    for (int k = 0; k < kRpt; ++k) {
        const int r = rb * Geo::kBlockRows + k * kRows + rsub;  // row of tile x
        const int g = r / T, t = r - g * T;
        ok[k] = g < p.heads_per_cta && x * T + t < job.z;
        slot0[k] = x * kM + r;
        M[k] = -INFINITY;
        L[k] = 0.f;
        A[k][0] = A[k][1] = A[k][2] = A[k][3] = 0.f;
    }
    // Fold one state (m, l, o) into (M, L, A): the online rule.
    auto fold = [](float &Mk, float &Lk, float *Ak, float m, float l, float o0, float o1, float o2, float o3) {
        if (m == -INFINITY)
            return;  // an empty piece (no visible token): weight 0
        if (m > Mk) {
            const float alpha = ex2(Mk - m);  // 0 while M is -inf
            Lk *= alpha;
            Ak[0] *= alpha;
            Ak[1] *= alpha;
            Ak[2] *= alpha;
            Ak[3] *= alpha;
            Mk = m;
        }
        const float wgt = m == Mk ? 1.f : ex2(m - Mk);
        Lk += wgt * l;
        Ak[0] += wgt * o0;
        Ak[1] += wgt * o1;
        Ak[2] += wgt * o2;
        Ak[3] += wgt * o3;
    };
    for (int cc = c + q; cc <= job.x; cc += Q) {
        const int base = (cc * 2 + (cc == c ? 1 : 0)) * 2 * kM;  // slot (cc, 1 or 0), tile 0, row 0
        float2 ml[kRpt];
        float4 v[kRpt];
#pragma unroll
        for (int k = 0; k < kRpt; ++k)
            if (ok[k]) {
                ml[k] = __ldcg(&p.part_ml[base + slot0[k]]);
                v[k] = __ldcg(reinterpret_cast<const float4 *>(p.part_o + (size_t)(base + slot0[k]) * D) + tpr);
            }
#pragma unroll
        for (int k = 0; k < kRpt; ++k)
            if (ok[k])
                fold(M[k], L[k], A[k], ml[k].x, ml[k].y, v[k].x, v[k].y, v[k].z, v[k].w);
    }
    if constexpr (Q > 1) {
        // Planes 1 .. Q-1 hand their states to plane 0, which folds them in order.
        float *st = s_st + ((rsub * Q + q) * kTpr + tpr) * 6;
        st[0] = M[0];
        st[1] = L[0];
        st[2] = A[0][0];
        st[3] = A[0][1];
        st[4] = A[0][2];
        st[5] = A[0][3];
        __syncthreads();
        if (q != 0)
            return;
#pragma unroll 1
        for (int qq = 1; qq < Q; ++qq) {
            const float *o = s_st + ((rsub * Q + qq) * kTpr + tpr) * 6;
            fold(M[0], L[0], A[0], o[0], o[1], o[2], o[3], o[4], o[5]);
        }
    }
#pragma unroll
    for (int k = 0; k < kRpt; ++k) {
        if (!ok[k])
            continue;
        const int r = rb * Geo::kBlockRows + k * kRows + rsub;
        const int g = r / T, t = r - g * T;
        const float inv = L[k] > 0.f ? p.v_scale / L[k] : 0.f;
        uint16_t *out = static_cast<uint16_t *>(p.out) +
                        ((long long)(job.y + x * T + t) * p.num_q_heads + job.w + g) * D + tpr * 4;
        *reinterpret_cast<uint2 *>(out) =
            make_uint2(pack2<BF16>(A[k][0] * inv, A[k][1] * inv), pack2<BF16>(A[k][2] * inv, A[k][3] * inv));
    }
}

// ================================================================ host side

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Pool as rank 5 (head_size, kv_heads, block slots, blocks, K|V), box of 64
// dims x one head x 16 slots x one block x one of K/V: 2 KB, 128-byte swizzle.
int encode_kv_map(CUtensorMap *m, const void *kv, int num_blocks, int block_size, int num_kv_heads, int d)
{
    const cuuint64_t e = 2, hd = (cuuint64_t)d;
    cuuint64_t dims[5] = {hd, (cuuint64_t)num_kv_heads, (cuuint64_t)block_size, (cuuint64_t)num_blocks, 2};
    cuuint64_t strides[4] = {hd * e, (cuuint64_t)num_kv_heads * hd * e,
                             (cuuint64_t)block_size * num_kv_heads * hd * e,
                             (cuuint64_t)num_blocks * block_size * num_kv_heads * hd * e};
    cuuint32_t box[5] = {64, 1, (cuuint32_t)kBoxTokens, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, const_cast<void *>(kv), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : set_error(PA_ERR_CUDA, "pa_prefill: K/V tensor map (%d)", (int)r);
}

// An FP8 pool as rank 5 (head_size bytes, kv_heads, block slots, blocks,
// K|V), box of the d codes of one head x 16 slots: 128-byte rows with the
// 128-byte swizzle at d = 128 (2 KB), plain 64-byte rows at d = 64 (1 KB).
int encode_kv_map_fp8(CUtensorMap *m, const void *kv, int num_blocks, int block_size, int num_kv_heads, int d)
{
    const cuuint64_t hd = (cuuint64_t)d;
    cuuint64_t dims[5] = {hd, (cuuint64_t)num_kv_heads, (cuuint64_t)block_size, (cuuint64_t)num_blocks, 2};
    cuuint64_t strides[4] = {hd, (cuuint64_t)num_kv_heads * hd, (cuuint64_t)block_size * num_kv_heads * hd,
                             (cuuint64_t)num_blocks * block_size * num_kv_heads * hd};
    cuuint32_t box[5] = {(cuuint32_t)d, 1, (cuuint32_t)kBoxTokens, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(kv), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           d == kD ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : set_error(PA_ERR_CUDA, "pa_prefill_fp8: K/V tensor map (%d)", (int)r);
}

// Queries as rank 3 (head_size, q_heads, tokens), box of 64 dims x one head x
// rows_per_head tokens.
int encode_q_map(CUtensorMap *m, const void *q, int total_q, int num_q_heads, int rows, int d)
{
    const cuuint64_t e = 2, hd = (cuuint64_t)d;
    cuuint64_t dims[3] = {hd, (cuuint64_t)num_q_heads, (cuuint64_t)total_q};
    cuuint64_t strides[2] = {hd * e, (cuuint64_t)num_q_heads * hd * e};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(q), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : set_error(PA_ERR_CUDA, "pa_prefill: query tensor map (%d)", (int)r);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int prefill_take_device_error(int *bits)
{
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof(int));
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(int));
    *bits = e == cudaSuccess ? v : 0;
    return (int)e;
}

}  // namespace pa

using namespace pa;

namespace {

// A launch's work units and scheduling. With enough units, each of
// min(units, SMs) persistent CTAs takes whole units, heaviest first, from a
// counter. With few (at most kSplitUnitsPerSm per SM, and a workspace), the
// units' K/V tiles are dealt out in equal contiguous shares (stream-K) to
// one CTA per SM, however many pieces that cuts a unit into (the merge
// spreads a unit's pieces over several threads per row).
constexpr int kSplitUnitsPerSm = 4;

struct LaunchPlan {
    int heads_per_cta, head_tiles, rows_per_head, q_pairs;
    long long units;
    int split_grid;     // G under stream-K, 0 when the launch takes whole units
    size_t split_bytes; // workspace stream-K needs
};

LaunchPlan plan_launch(int num_seqs, int max_seqlen_q, int num_q_heads, int num_kv_heads, int head_size, int sms)
{
    LaunchPlan lp;
    const int group = num_q_heads / num_kv_heads;
    lp.heads_per_cta = group < 16 ? group : 16;
    lp.head_tiles = group / lp.heads_per_cta;
    lp.rows_per_head = (kM / lp.heads_per_cta) & ~7;
    const int q_tiles = (max_seqlen_q + lp.rows_per_head - 1) / lp.rows_per_head;
    lp.q_pairs = (q_tiles + 1) / 2;
    lp.units = (long long)lp.q_pairs * num_seqs * num_kv_heads * lp.head_tiles;
    lp.split_grid = 0;
    lp.split_bytes = 0;
    if (lp.units > 0 && lp.units <= std::min<long long>(kMaxSplitUnits, (long long)kSplitUnitsPerSm * sms)) {
        lp.split_grid = sms;
        // Per CTA two slots of two 128-row tiles: O rows (head_size fp32)
        // and (m, l) pairs; then one job record per CTA.
        lp.split_bytes = (size_t)lp.split_grid * 2 * 2 * kM * ((size_t)head_size * 4 + 8) + (size_t)lp.split_grid * 16;
    }
    return lp;
}

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous one in the stream finishes and waits for it with
// griddepcontrol.wait before reading what it wrote.
cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, void **args, size_t smem, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// SM count of the current device (cached per device).
int current_sms(const char *who, int *dev_out, int *sms_out)
{
    static std::mutex mu;
    static int sm_count[64] = {};
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return set_error(PA_ERR_CUDA, "%s: cudaGetDevice: %s", who, cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(mu);
    sms = dev < 64 ? sm_count[dev] : 0;
    if (sms <= 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess || sms <= 0)
            return set_error(PA_ERR_CUDA, "%s: SM count: %s", who, cudaGetErrorString(e));
        if (dev < 64)
            sm_count[dev] = sms;
    }
    *dev_out = dev;
    *sms_out = sms;
    return PA_OK;
}

int check_heads(const char *who, int num_q_heads, int num_kv_heads, int head_size)
{
    if (head_size != kD && head_size != 64)
        return set_error(PA_ERR_UNSUPPORTED, "%s: head_size %d (built: 64 and 128)", who, head_size);
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return set_error(PA_ERR_INVALID_ARG,
                         "%s: num_q_heads %d must be a positive multiple of num_kv_heads %d", who,
                         num_q_heads, num_kv_heads);
    const int group = num_q_heads / num_kv_heads;
    if (group > 16 && group % 16 != 0)
        return set_error(PA_ERR_UNSUPPORTED, "%s: query group %d (want <= 16 or a multiple of 16)", who,
                         group);
    return PA_OK;
}

int prefill_impl(const char *who, void *out, const void *query, const void *kv_cache, const int32_t *block_tables,
                 int max_blocks_per_seq, const int32_t *cu_seqlens_q, const int32_t *seq_lens, int num_seqs,
                 int total_q, int max_seqlen_q, float scale, int num_q_heads, int num_kv_heads, int head_size,
                 int num_blocks, int block_size, int dtype, bool fp8, float k_scale, float v_scale,
                 void *workspace, size_t workspace_bytes, pa_stream_t stream)
{
    if (dtype != PA_F16 && dtype != PA_BF16)
        return set_error(PA_ERR_UNSUPPORTED, "%s: dtype %d (want PA_F16 or PA_BF16)", who, dtype);
    int rc = check_heads(who, num_q_heads, num_kv_heads, head_size);
    if (rc != PA_OK)
        return rc;
    const int group = num_q_heads / num_kv_heads;
    if (block_size < kBoxTokens || block_size % kBoxTokens != 0)
        return set_error(PA_ERR_INVALID_ARG, "%s: block_size %d must be a positive multiple of 16", who,
                         block_size);
    if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
        return set_error(PA_ERR_INVALID_ARG, "%s: bad sizes", who);
    if ((long long)max_blocks_per_seq * block_size > (1LL << 30))
        return set_error(PA_ERR_INVALID_ARG, "%s: max_blocks_per_seq * block_size too large", who);
    if (!std::isfinite(scale))
        return set_error(PA_ERR_INVALID_ARG, "%s: scale is not finite", who);
    if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0)
        return PA_OK;
    if (!out || !query || !kv_cache || !block_tables || !cu_seqlens_q || !seq_lens)
        return set_error(PA_ERR_INVALID_ARG, "%s: null pointer argument", who);
    if (!aligned16(out) || !aligned16(query) || !aligned16(kv_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3) || (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3))
        return set_error(PA_ERR_INVALID_ARG, "%s: misaligned pointer (query/out/pool 16 B)", who);
    if (!encoder())
        return set_error(PA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");

    int dev = 0, sms = 0;
    rc = current_sms(who, &dev, &sms);
    if (rc != PA_OK)
        return rc;
    const LaunchPlan lp = plan_launch(num_seqs, max_seqlen_q, num_q_heads, num_kv_heads, head_size, sms);
    if (lp.units > 0x7fffffffLL)
        return set_error(PA_ERR_UNSUPPORTED, "%s: too many query tiles", who);
    // Stream-K needs the workspace; without one the launch takes whole units.
    const bool split = lp.split_grid > 0 && workspace != nullptr;
    if (split && (workspace_bytes < lp.split_bytes || (reinterpret_cast<uintptr_t>(workspace) & 255)))
        return set_error(PA_ERR_WORKSPACE, "%s: workspace of %zu bytes at %p (need %zu, 256-byte aligned)", who,
                         workspace_bytes, workspace, lp.split_bytes);

    PrefillParams prm;
    prm.out = out;
    prm.block_tables = block_tables;
    prm.cu_q = cu_seqlens_q;
    prm.seq_lens = seq_lens;
    prm.max_blocks_per_seq = max_blocks_per_seq;
    prm.num_seqs = num_seqs;
    prm.num_q_heads = num_q_heads;
    prm.group = group;
    prm.heads_per_cta = lp.heads_per_cta;
    prm.head_tiles = lp.head_tiles;
    prm.rows_per_head = lp.rows_per_head;
    prm.q_pairs = lp.q_pairs;
    prm.max_q = max_seqlen_q;
    prm.num_blocks = num_blocks;
    prm.block_size = block_size;
    prm.total_q = total_q;
    prm.max_len = max_blocks_per_seq * block_size;
    prm.scale_log2 = scale * 1.4426950408889634f * (fp8 ? k_scale : 1.f);
    prm.v_scale = fp8 ? v_scale : 1.f;
    prm.num_kv_heads = num_kv_heads;
    prm.num_units = (int)lp.units;
    prm.part_o = split ? static_cast<float *>(workspace) : nullptr;
    prm.part_ml = split ? reinterpret_cast<float2 *>(static_cast<float *>(workspace) +
                                                     (size_t)lp.split_grid * 2 * 2 * kM * head_size)
                        : nullptr;
    prm.jobs = split ? reinterpret_cast<int4 *>(prm.part_ml + (size_t)lp.split_grid * 2 * 2 * kM) : nullptr;
    static std::atomic<unsigned> launches{0};
    prm.sched_slot = (int)(launches.fetch_add(1u) % (unsigned)kSchedSlots);

    CUtensorMap kv_map, q_map;
    rc = fp8 ? encode_kv_map_fp8(&kv_map, kv_cache, num_blocks, block_size, num_kv_heads, head_size)
                 : encode_kv_map(&kv_map, kv_cache, num_blocks, block_size, num_kv_heads, head_size);
    if (rc != PA_OK)
        return rc;
    rc = encode_q_map(&q_map, query, total_q, num_q_heads, prm.rows_per_head, head_size);
    if (rc != PA_OK)
        return rc;

    const bool bf = dtype == PA_BF16, d64 = head_size == 64;
    // Instances by (stream-K, FP8 cache, head size 64, bf16).
#define PA_PREFILL_INSTANCES(SK)                                                              \
    reinterpret_cast<const void *>(&paged_prefill_kernel<false, false, 128, SK>),               \
        reinterpret_cast<const void *>(&paged_prefill_kernel<true, false, 128, SK>),           \
        reinterpret_cast<const void *>(&paged_prefill_kernel<false, false, 64, SK>),           \
        reinterpret_cast<const void *>(&paged_prefill_kernel<true, false, 64, SK>),            \
        reinterpret_cast<const void *>(&paged_prefill_kernel<false, true, 128, SK>),           \
        reinterpret_cast<const void *>(&paged_prefill_kernel<true, true, 128, SK>),            \
        reinterpret_cast<const void *>(&paged_prefill_kernel<false, true, 64, SK>),            \
        reinterpret_cast<const void *>(&paged_prefill_kernel<true, true, 64, SK>)
    static const void *const kernels[16] = {PA_PREFILL_INSTANCES(false), PA_PREFILL_INSTANCES(true)};
#undef PA_PREFILL_INSTANCES
    const int variant = (split ? 8 : 0) + (fp8 ? 4 : 0) + (d64 ? 2 : 0) + (bf ? 1 : 0);
    const void *fn = kernels[variant];
    // Raise the kernel's shared-memory limit once per device (a call being
    // captured into a CUDA graph then makes no attribute call; the SM count
    // is cached likewise).
    static std::mutex mu;
    static bool raised[16][64] = {};
    cudaError_t e;
    {
        std::lock_guard<std::mutex> lock(mu);
        bool &done = raised[variant][dev & 63];
        if (!done) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess)
                return set_error(PA_ERR_CUDA, "%s: cudaFuncSetAttribute: %s", who, cudaGetErrorString(e));
            done = dev < 64;
        }
    }
    // Persistent grid: one CTA per SM (the CTA holds 225 KB of shared
    // memory), never more CTAs than units; G CTAs under stream-K.
    const dim3 grid(split ? (unsigned)lp.split_grid : (unsigned)std::min<long long>(lp.units, sms));
    void *args[] = {&kv_map, &q_map, &prm};
    e = cudaLaunchKernel(fn, grid, dim3(threads_for(fp8)), args, kSmemBytes, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return set_error(PA_ERR_CUDA, "%s: launch: %s", who, cudaGetErrorString(e));
    if (split) {
        // Merge planes: enough that each thread folds about 8 pieces of a
        // unit cut into G / units + 1 pieces.
        const long long pieces = ((long long)lp.split_grid + lp.units - 1) / lp.units + 1;
        const int qi = pieces <= 8 ? 0 : pieces <= 16 ? 1 : pieces <= 32 ? 2 : 3;
#define PA_MERGE_INSTANCES(Q)                                                                      \
    reinterpret_cast<const void *>(&paged_prefill_merge_kernel<false, 128, Q>),                    \
        reinterpret_cast<const void *>(&paged_prefill_merge_kernel<true, 128, Q>),                 \
        reinterpret_cast<const void *>(&paged_prefill_merge_kernel<false, 64, Q>),                 \
        reinterpret_cast<const void *>(&paged_prefill_merge_kernel<true, 64, Q>)
        static const void *const merges[16] = {PA_MERGE_INSTANCES(1), PA_MERGE_INSTANCES(2), PA_MERGE_INSTANCES(4),
                                               PA_MERGE_INSTANCES(8)};
#undef PA_MERGE_INSTANCES
        static const int blocks128[4] = {MergeGeo<128, 1>::kBlocks, MergeGeo<128, 2>::kBlocks,
                                         MergeGeo<128, 4>::kBlocks, MergeGeo<128, 8>::kBlocks};
        static const int blocks64[4] = {MergeGeo<64, 1>::kBlocks, MergeGeo<64, 2>::kBlocks, MergeGeo<64, 4>::kBlocks,
                                        MergeGeo<64, 8>::kBlocks};
        int grid_main = lp.split_grid;
        const long long jobs = std::min<long long>(lp.units, grid_main);  // at most one per unit and per CTA
        const int merge_grid = (int)(jobs * 2 * (d64 ? blocks64[qi] : blocks128[qi]));
        void *margs[] = {&prm, &grid_main};
        e = launch_pdl(merges[qi * 4 + (d64 ? 2 : 0) + (bf ? 1 : 0)], dim3(merge_grid), dim3(256), margs, 0,
                       reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess)
            return set_error(PA_ERR_CUDA, "%s: merge launch: %s", who, cudaGetErrorString(e));
    }
    return PA_OK;
}

}  // namespace

extern "C" int pa_prefill(void *out, const void *query, const void *kv_cache, const int32_t *block_tables,
                          int max_blocks_per_seq, const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                          int num_seqs, int total_q, int max_seqlen_q, float scale, int num_q_heads,
                          int num_kv_heads, int head_size, int num_blocks, int block_size, int dtype,
                          void *workspace, size_t workspace_bytes, pa_stream_t stream)
{
    return prefill_impl("pa_prefill", out, query, kv_cache, block_tables, max_blocks_per_seq, cu_seqlens_q,
                        seq_lens, num_seqs, total_q, max_seqlen_q, scale, num_q_heads, num_kv_heads, head_size,
                        num_blocks, block_size, dtype, false, 1.f, 1.f, workspace, workspace_bytes, stream);
}

extern "C" int pa_prefill_fp8(void *out, const void *query, const void *kv_cache, const int32_t *block_tables,
                              int max_blocks_per_seq, const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                              int num_seqs, int total_q, int max_seqlen_q, float scale, int num_q_heads,
                              int num_kv_heads, int head_size, int num_blocks, int block_size, int dtype,
                              float k_scale, float v_scale, void *workspace, size_t workspace_bytes,
                              pa_stream_t stream)
{
    if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
        return set_error(PA_ERR_INVALID_ARG, "pa_prefill_fp8: k_scale and v_scale must be finite and > 0");
    return prefill_impl("pa_prefill_fp8", out, query, kv_cache, block_tables, max_blocks_per_seq, cu_seqlens_q,
                        seq_lens, num_seqs, total_q, max_seqlen_q, scale, num_q_heads, num_kv_heads, head_size,
                        num_blocks, block_size, dtype, true, k_scale, v_scale, workspace, workspace_bytes, stream);
}

extern "C" int pa_prefill_workspace_size(int num_seqs, int max_seqlen_q, int num_q_heads, int num_kv_heads,
                                         int head_size, size_t *bytes)
{
    const char *who = "pa_prefill_workspace_size";
    if (!bytes)
        return set_error(PA_ERR_INVALID_ARG, "%s: null bytes", who);
    *bytes = 0;
    int rc = check_heads(who, num_q_heads, num_kv_heads, head_size);
    if (rc != PA_OK)
        return rc;
    if (num_seqs < 0 || max_seqlen_q < 0)
        return set_error(PA_ERR_INVALID_ARG, "%s: bad sizes", who);
    if (num_seqs == 0 || max_seqlen_q == 0)
        return PA_OK;
    int dev = 0, sms = 0;
    rc = current_sms(who, &dev, &sms);
    if (rc != PA_OK)
        return rc;
    *bytes = plan_launch(num_seqs, max_seqlen_q, num_q_heads, num_kv_heads, head_size, sms).split_bytes;
    return PA_OK;
}
