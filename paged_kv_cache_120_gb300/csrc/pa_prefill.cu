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
// How it is computed (one CTA = 128 query rows of one (sequence, kv head)):
//  * Rows are (query head of the kv head's group, query token) pairs, so the
//    heads that share a kv head share every K/V tile. A TMEM lane per row.
//  * Warp 8 loads Q once and the K tiles, warp 10 the V tiles, by TMA
//    (16-token boxes looked up through the block table, 128-byte swizzle),
//    into rings of three K and two V stages, each at its own pace. One
//    thread of warp 9 issues the MMAs: S = Q K^T into one of two TMEM
//    buffers, then O += P V (V read as an MN-major operand) into a third,
//    so the next tile's scores overlap this tile's softmax.
//  * Warps 0-7 run the softmax, two warps per row: warp w and w + 4 share
//    the TMEM lanes of row quarter w % 4 and take the row's columns 0-63 and
//    64-127. Each scales and masks its half causally, the two swap partial
//    maxima through TMEM, and both run the same fp32 online softmax in base
//    2 (the reference maximum moves only when a score exceeds it by 2^8, so
//    O in TMEM is rarely rescaled and the next tile's softmax need not wait
//    for this tile's P V), writing their half of P (rounded to the element
//    type) to shared memory in the MMA's swizzled layout. Two warps per
//    row keep two softmax warps issuing on every SM sub-partition. At the
//    end the partial row sums meet, and each warp divides and stores its
//    half of O.
//  * Every wait is bounded; the K/V rows past a sequence's end (padding slots
//    of its last block, possibly NaN) are zeroed before P V reads them.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__device__ int g_prefill_error;  // PA_DEVERR_* bits of the prefill kernels

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

// One fp32 column of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tc_st1(uint32_t taddr, float v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "f"(v) : "memory");
}

__device__ __forceinline__ float tc_ld1(uint32_t taddr)
{
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    return __uint_as_float(r);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// ----------------------------------------------------------------- layout

constexpr int kD = 128;                    // head size (the one built)
constexpr int kM = 128;                    // query rows per CTA (TMEM lanes)
constexpr int kN = 128;                    // cached tokens per K/V tile
constexpr int kChunkBytes = 128 * 128;     // a 64-column, 128-row swizzled chunk: 16 KB
constexpr int kTileBytes = 2 * kChunkBytes;  // a 128 x 128 16-bit operand: 32 KB
constexpr int kBoxTokens = 16;             // tokens per K/V TMA box (block_size is a multiple)
constexpr int kThreads = 352;              // warps 0-7 softmax, 8 Q/K TMA, 9 MMA, 10 V TMA
constexpr int kSoftmaxThreads = 256;       // two warps per row quarter, one per 64-column half
constexpr int kWarpQK = 8, kWarpMMA = 9, kWarpV = 10;
constexpr int kKStages = 3;                // K ring (freed when S = Q K^T is done)
constexpr int kVStages = 2;                // V ring (freed when O += P V is done)
constexpr int kOffQ = 0;
constexpr int kOffK = kTileBytes;
constexpr int kOffV = kOffK + kKStages * kTileBytes;
constexpr int kOffP = kOffV + kVStages * kTileBytes;
constexpr int kSmemBytes = kOffP + kTileBytes + 1024;  // + slack to align the base to 1024
constexpr uint32_t kTmemCols = 512;        // S (two buffers) and O, 128 columns each, + exchange
constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO = 256;
constexpr uint32_t kTmemX = 384;           // row maxima (2 parities x 2 halves) and row sums (2 halves)
constexpr float kRescaleLog2 = 8.f;        // reference-maximum slack (base 2)

struct PrefillParams {
    void *out;
    const int32_t *block_tables;
    const int32_t *cu_q;
    const int32_t *seq_lens;
    int max_blocks_per_seq;
    int num_seqs;
    int num_q_heads;
    int group;          // num_q_heads / num_kv_heads
    int heads_per_cta;  // query heads of one kv head that share a CTA (<= 16)
    int head_tiles;     // group / heads_per_cta
    int rows_per_head;  // query tokens per CTA (multiple of 8)
    int q_tiles;        // ceil(max_seqlen_q / rows_per_head)
    int num_blocks;
    int block_size;
    int total_q;
    int max_len;        // max_blocks_per_seq * block_size
    float scale_log2;   // scale * log2(e)
};

struct PrefillBars {
    uint64_t q_full, k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2], p_full, pv_done;
    uint64_t xch[4];  // per row quarter: the two half-row warps exchanged their values
    uint32_t tmem_base;
    int fail;
};

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap kv_map,
                         const __grid_constant__ CUtensorMap q_map, const PrefillParams p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ PrefillBars bars;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.z, h = blockIdx.y;
    const int ht = blockIdx.x % p.head_tiles;
    const int qt = (p.q_tiles - 1) - blockIdx.x / p.head_tiles;  // heaviest tiles start first
    const int T = p.rows_per_head, HPC = p.heads_per_cta;

    // The unit (uniform across the CTA); bad offsets or lengths are flagged
    // by the first CTA of the sequence and skipped.
    const int q0 = p.cu_q[s];
    const int q_len = p.cu_q[s + 1] - q0;
    const int L = p.seq_lens[s];
    if (q_len < 0 || q0 < 0 || q0 + q_len > p.total_q || L < q_len || L > p.max_len) {
        if (tid == 0 && blockIdx.x == 0 && h == 0)
            prefill_raise(PA_DEVERR_SEQ_LEN);
        return;
    }
    const int t0 = qt * T;
    if (t0 >= q_len)
        return;
    const int t_end = min(q_len, t0 + T);
    const int n_tiles = (L - q_len + t_end + kN - 1) / kN;  // tiles the tile's last query sees

    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sQ = base + kOffQ, sP = base + kOffP;
    auto sK = [&](int st) { return base + kOffK + st * kTileBytes; };
    auto sV = [&](int st) { return base + kOffV + st * kTileBytes; };
    const uint32_t b_q = smem_addr(&bars.q_full), b_p = smem_addr(&bars.p_full),
                   b_pv = smem_addr(&bars.pv_done);
    auto b_kf = [&](int st) { return smem_addr(&bars.k_full[st]); };
    auto b_ke = [&](int st) { return smem_addr(&bars.k_empty[st]); };
    auto b_vf = [&](int st) { return smem_addr(&bars.v_full[st]); };
    auto b_ve = [&](int st) { return smem_addr(&bars.v_empty[st]); };
    auto b_s = [&](int b) { return smem_addr(&bars.s_full[b]); };

    if (tid == 0) {
        mbar_init(b_q, 1);
        for (int st = 0; st < kKStages; ++st) {
            mbar_init(b_kf(st), 1);
            mbar_init(b_ke(st), 1);
        }
        for (int st = 0; st < kVStages; ++st) {
            mbar_init(b_vf(st), 1);
            mbar_init(b_ve(st), 1);
        }
        mbar_init(b_s(0), 1);
        mbar_init(b_s(1), 1);
        mbar_init(b_p, kSoftmaxThreads);
        mbar_init(b_pv, 1);
        for (int i = 0; i < 4; ++i)
            mbar_init(smem_addr(&bars.xch[i]), 64);
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

    // Give up on a wait that runs out (recorded once per CTA); every role then
    // drains to the teardown.
    auto wait_or_fail = [&](uint32_t bar, uint32_t parity) {
        if (mbar_wait(bar, parity))
            return true;
        if (atomicExch(&bars.fail, 1) == 0)
            prefill_raise(PA_DEVERR_TIMEOUT);
        return false;
    };

    if (warp == kWarpQK || warp == kWarpV) {
        // ---------------------------------------------------------- TMA
        // Warp 4 produces Q and the K tiles, warp 6 the V tiles, each at its
        // own pace (separate warps, so that one producer's wait never holds
        // up the other); lane i < 8 moves the 16-token box i of each tile.
        // The block-table entry of the next tile is loaded while the current
        // one waits for its stage.
        const int32_t *table = p.block_tables + (long long)s * p.max_blocks_per_seq;
        const bool is_k = warp == kWarpQK;
        if (is_k && lane == 0) {
            const int head0 = h * p.group + ht * HPC;
            mbar_expect_tx(b_q, (uint32_t)(2 * HPC * T * 128));
            for (int c = 0; c < 2; ++c)
                for (int g = 0; g < HPC; ++g)
                    tma_load_3d(sQ + c * kChunkBytes + g * T * 128, &q_map, b_q, c * 64, head0 + g, q0 + t0);
        }
        if (lane < 8) {
            const int box = lane, leader = 0;
            const unsigned group_mask = 0x000000FFu;
            const int stages = is_k ? kKStages : kVStages;
            auto lookup = [&](int j) {
                const int kt = j * kN + kBoxTokens * box;
                return (j < n_tiles && kt < L) ? __ldg(table + kt / p.block_size) : -1;
            };
            int next = lookup(0);
            for (int j = 0; j < n_tiles; ++j) {
                int phys = next;
                next = lookup(j + 1);
                const int st = j % stages;
                if (j >= stages &&
                    !wait_or_fail(is_k ? b_ke(st) : b_ve(st), ((j - stages) / stages) & 1))
                    break;
                const int kt = j * kN + kBoxTokens * box;
                const int tib = kt % p.block_size;
                if (phys >= p.num_blocks || (phys < 0 && kt < L)) {
                    prefill_raise(PA_DEVERR_BLOCK_ID);
                    phys = p.num_blocks;
                }
                if (phys < 0)
                    phys = p.num_blocks;  // past the sequence end: outside the map, zeros
                const uint32_t full = is_k ? b_kf(st) : b_vf(st);
                if (lane == leader)
                    mbar_expect_tx(full, kTileBytes);
                __syncwarp(group_mask);
                const uint32_t dst = (is_k ? sK(st) : sV(st)) + box * (kBoxTokens * 128);
                for (int c = 0; c < 2; ++c)
                    tma_load_5d(dst + c * kChunkBytes, &kv_map, full, c * 64, h, tib, phys, is_k ? 0 : 1);
            }
        }
    } else if (warp == kWarpMMA) {
        // ---------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t id_s = instr_desc(kM, kN, BF16, false);
            const uint32_t id_o = instr_desc(kM, kD, BF16, true);
            auto issue_pv = [&](int jj) {
                const int vs = jj % kVStages;
                if (!wait_or_fail(b_p, jj & 1) || !wait_or_fail(b_vf(vs), (jj / kVStages) & 1))
                    return false;
                tc_fence_after();
                // O += P V: A = P (K-major over tokens), B = V (MN-major:
                // 64-dim chunks 16 KB apart, 8-token groups 1 KB apart).
                for (int k = 0; k < kN / 16; ++k)
                    tc_mma(tmem + kTmemO, smem_desc(sP + (k >> 2) * kChunkBytes + (k & 3) * 32, 16, 1024),
                           smem_desc(sV(vs) + k * 2048, kChunkBytes, 1024), id_o,
                           (jj > 0 || k > 0) ? 1u : 0u);
                tc_commit(b_pv);
                tc_commit(b_ve(vs));
                return true;
            };
            bool go = wait_or_fail(b_q, 0);
            for (int j = 0; go && j < n_tiles; ++j) {
                const int ks = j % kKStages;
                if (!wait_or_fail(b_kf(ks), (j / kKStages) & 1))
                    break;
                tc_fence_after();
                // S = Q K^T over the head dimension, 16 per MMA.
                const uint32_t tS = tmem + ((j & 1) ? kTmemS1 : kTmemS0);
                for (int k = 0; k < kD / 16; ++k) {
                    const uint32_t off = (k >> 2) * kChunkBytes + (k & 3) * 32;
                    tc_mma(tS, smem_desc(sQ + off, 16, 1024), smem_desc(sK(ks) + off, 16, 1024), id_s,
                           k > 0 ? 1u : 0u);
                }
                tc_commit(b_s(j & 1));
                tc_commit(b_ke(ks));
                if (j > 0)
                    go = issue_pv(j - 1);
            }
            if (go)
                issue_pv(n_tiles - 1);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------- softmax (half rows)
        // Warps w and w + 4 share the TMEM lanes of row quarter w % 4 (a
        // warp may only touch its quarter); warp w takes columns 0-63 of
        // each row, warp w + 4 columns 64-127. They swap their partial row
        // maxima (and at the end their partial row sums) through TMEM
        // columns kTmemX.., with a per-quarter mbarrier in between, so both
        // take identical rescaling decisions.
        const int quarter = warp & 3, hf = warp >> 2;
        const int r = quarter * 32 + lane;  // this thread's TMEM lane (row)
        const int g = r / T, t = r - g * T;
        const bool valid = g < HPC && t0 + t < q_len;
        const int pos = valid ? L - q_len + t0 + t : -1;  // last token this row sees
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t b_x = smem_addr(&bars.xch[quarter]);
        const int c0 = hf * 64;  // first column of this warp's half
        float m_run = -INFINITY, l_run = 0.f;
        bool alive = true;
        // Publish v in exchange column `col`, meet the partner warp (phase
        // `ph`), return the partner's value from column `col ^ 1`.
        auto swap = [&](uint32_t col, float v, uint32_t ph, float &other) {
            tc_st1(tmem + lane_off + col, v);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            mbar_arrive(b_x);
            if (!__all_sync(kFull, wait_or_fail(b_x, ph)))
                return false;
            tc_fence_after();
            other = tc_ld1(tmem + lane_off + (col ^ 1u));
            return true;
        };
        for (int j = 0; j < n_tiles; ++j) {
            const int b = j & 1;
            if (!__all_sync(kFull, wait_or_fail(b_s(b), (j >> 1) & 1))) {
                alive = false;
                break;
            }
            tc_fence_after();
            float sv[64];
            {
                const uint32_t tS = tmem + lane_off + (b ? kTmemS1 : kTmemS0) + c0;
                uint32_t *rawv = reinterpret_cast<uint32_t *>(sv);
                tc_ld32_async(tS, rawv);
                tc_ld32_async(tS + 32, rawv + 32);
                tc_wait_ld();
            }
            const int kbase = j * kN + c0;
            // Scale (and mask) the half row; its maximum over 8 chains.
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                m8[i] = -INFINITY;
            if (kbase + 63 <= pos) {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    sv[c] *= p.scale_log2;
                    m8[c & 7] = fmaxf(m8[c & 7], sv[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    sv[c] = (kbase + c <= pos) ? sv[c] * p.scale_log2 : -INFINITY;
                    m8[c & 7] = fmaxf(m8[c & 7], sv[c]);
                }
            }
            const float mh = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            float mo;
            if (!swap(kTmemX + 2 * b + hf, mh, b, mo)) {
                alive = false;
                break;
            }
            const float mx = fmaxf(mh, mo);
            // The row's reference maximum moves only when a score exceeds it
            // by more than kRescaleLog2 (P then stays <= 2^kRescaleLog2, which
            // the element type holds with full relative precision); O and l
            // are rescaled only then. Both halves see the same mx.
            const bool grow = mx > m_run + kRescaleLog2;
            const float m_new = grow ? mx : m_run;
            const float alpha = grow ? ex2(m_run - m_new) : 1.f;
            const float ref = m_new == -INFINITY ? 0.f : m_new;
            // P, rounded to the element type, packed in registers; the row
            // sum adds the same rounded values.
            uint32_t pw[32];
            float l8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                l8[i] = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                pw[c] = pack2<BF16>(ex2(sv[2 * c] - ref), ex2(sv[2 * c + 1] - ref));
                const float2 f = unpack2<BF16>(pw[c]);
                l8[c & 7] += f.x + f.y;
            }
            const float ls = ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
            // The previous tile's P V must be done before P is overwritten
            // and before O is rescaled.
            if (j > 0 && !__all_sync(kFull, wait_or_fail(b_pv, (j - 1) & 1))) {
                alive = false;
                break;
            }
            tc_fence_after();
            if (j > 0 && __any_sync(kFull, alpha != 1.f)) {
                const uint32_t tO = tmem + lane_off + kTmemO + c0;
                float o[32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    tc_ld32(tO + c * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] *= alpha;
                    tc_st32(tO + c * 32, o);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            // P into its K-major 128-byte swizzled rows: this half is the
            // 64-column chunk hf.
#pragma unroll
            for (int u = 0; u < 8; ++u)
                sts128(sP + hf * kChunkBytes + r * 128 + ((u ^ (r & 7)) << 4), pw[4 * u], pw[4 * u + 1],
                       pw[4 * u + 2], pw[4 * u + 3]);
            l_run = l_run * alpha + ls;
            m_run = m_new;
            // The last tile's V rows past the sequence end hold whatever the
            // pool's padding slots hold: zero them (P is 0 there) once V lands;
            // each half-row warp clears its 64-dim chunk of the row.
            if (j * kN + kN > L) {
                const int vs = j % kVStages;
                if (!__all_sync(kFull, wait_or_fail(b_vf(vs), (j / kVStages) & 1))) {
                    alive = false;
                    break;
                }
                if (j * kN + r >= L)
                    for (int u = 0; u < 8; ++u)
                        sts128(sV(vs) + hf * kChunkBytes + r * 128 + u * 16, 0u, 0u, 0u, 0u);
            }
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(b_p);
        }
        // Epilogue: the two partial row sums meet, then each warp stores its
        // 64 output columns, O / l, for the valid rows.
        float lo = 0.f;
        if (alive && swap(kTmemX + 4 + hf, l_run, (uint32_t)(n_tiles & 1), lo) &&
            __all_sync(kFull, wait_or_fail(b_pv, (n_tiles - 1) & 1))) {
            tc_fence_after();
            const float l_tot = l_run + lo;
            const uint32_t tO = tmem + lane_off + kTmemO + c0;
            const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
            uint16_t *out = static_cast<uint16_t *>(p.out) +
                            ((long long)(q0 + t0 + t) * p.num_q_heads + h * p.group + ht * HPC + g) * kD + c0;
            float o[32];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                tc_ld32(tO + c * 32, o);
                if (valid) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 v;
                        v.x = pack2<BF16>(o[8 * q + 0] * inv, o[8 * q + 1] * inv);
                        v.y = pack2<BF16>(o[8 * q + 2] * inv, o[8 * q + 3] * inv);
                        v.z = pack2<BF16>(o[8 * q + 4] * inv, o[8 * q + 5] * inv);
                        v.w = pack2<BF16>(o[8 * q + 6] * inv, o[8 * q + 7] * inv);
                        reinterpret_cast<uint4 *>(out + c * 32)[q] = v;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMMA)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
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
int encode_kv_map(CUtensorMap *m, const void *kv, int num_blocks, int block_size, int num_kv_heads)
{
    const cuuint64_t e = 2;
    cuuint64_t dims[5] = {(cuuint64_t)kD, (cuuint64_t)num_kv_heads, (cuuint64_t)block_size,
                          (cuuint64_t)num_blocks, 2};
    cuuint64_t strides[4] = {kD * e, (cuuint64_t)num_kv_heads * kD * e,
                             (cuuint64_t)block_size * num_kv_heads * kD * e,
                             (cuuint64_t)num_blocks * block_size * num_kv_heads * kD * e};
    cuuint32_t box[5] = {64, 1, (cuuint32_t)kBoxTokens, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, const_cast<void *>(kv), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : set_error(PA_ERR_CUDA, "pa_prefill: K/V tensor map (%d)", (int)r);
}

// Queries as rank 3 (head_size, q_heads, tokens), box of 64 dims x one head x
// rows_per_head tokens.
int encode_q_map(CUtensorMap *m, const void *q, int total_q, int num_q_heads, int rows)
{
    const cuuint64_t e = 2;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)num_q_heads, (cuuint64_t)total_q};
    cuuint64_t strides[2] = {kD * e, (cuuint64_t)num_q_heads * kD * e};
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

extern "C" int pa_prefill(void *out, const void *query, const void *kv_cache, const int32_t *block_tables,
                          int max_blocks_per_seq, const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                          int num_seqs, int total_q, int max_seqlen_q, float scale, int num_q_heads,
                          int num_kv_heads, int head_size, int num_blocks, int block_size, int dtype,
                          pa_stream_t stream)
{
    if (dtype != PA_F16 && dtype != PA_BF16)
        return set_error(PA_ERR_UNSUPPORTED, "pa_prefill: dtype %d (want PA_F16 or PA_BF16)", dtype);
    if (head_size != kD)
        return set_error(PA_ERR_UNSUPPORTED, "pa_prefill: head_size %d (built: 128)", head_size);
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return set_error(PA_ERR_INVALID_ARG,
                         "pa_prefill: num_q_heads %d must be a positive multiple of num_kv_heads %d",
                         num_q_heads, num_kv_heads);
    const int group = num_q_heads / num_kv_heads;
    if (group > 16 && group % 16 != 0)
        return set_error(PA_ERR_UNSUPPORTED, "pa_prefill: query group %d (want <= 16 or a multiple of 16)",
                         group);
    if (block_size < kBoxTokens || block_size % kBoxTokens != 0)
        return set_error(PA_ERR_INVALID_ARG, "pa_prefill: block_size %d must be a positive multiple of 16",
                         block_size);
    if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
        return set_error(PA_ERR_INVALID_ARG, "pa_prefill: bad sizes");
    if (num_seqs > 65535 || num_kv_heads > 65535)
        return set_error(PA_ERR_UNSUPPORTED, "pa_prefill: num_seqs and num_kv_heads must be <= 65535");
    if ((long long)max_blocks_per_seq * block_size > (1LL << 30))
        return set_error(PA_ERR_INVALID_ARG, "pa_prefill: max_blocks_per_seq * block_size too large");
    if (!std::isfinite(scale))
        return set_error(PA_ERR_INVALID_ARG, "pa_prefill: scale is not finite");
    if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0)
        return PA_OK;
    if (!out || !query || !kv_cache || !block_tables || !cu_seqlens_q || !seq_lens)
        return set_error(PA_ERR_INVALID_ARG, "pa_prefill: null pointer argument");
    if (!aligned16(out) || !aligned16(query) || !aligned16(kv_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3) || (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3))
        return set_error(PA_ERR_INVALID_ARG, "pa_prefill: misaligned pointer (query/out/pool 16 B)");
    if (!encoder())
        return set_error(PA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");

    PrefillParams prm;
    prm.out = out;
    prm.block_tables = block_tables;
    prm.cu_q = cu_seqlens_q;
    prm.seq_lens = seq_lens;
    prm.max_blocks_per_seq = max_blocks_per_seq;
    prm.num_seqs = num_seqs;
    prm.num_q_heads = num_q_heads;
    prm.group = group;
    prm.heads_per_cta = group < 16 ? group : 16;
    prm.head_tiles = group / prm.heads_per_cta;
    prm.rows_per_head = (kM / prm.heads_per_cta) & ~7;
    prm.q_tiles = (max_seqlen_q + prm.rows_per_head - 1) / prm.rows_per_head;
    prm.num_blocks = num_blocks;
    prm.block_size = block_size;
    prm.total_q = total_q;
    prm.max_len = max_blocks_per_seq * block_size;
    prm.scale_log2 = scale * 1.4426950408889634f;
    if ((long long)prm.q_tiles * prm.head_tiles > 0x7fffffffLL)
        return set_error(PA_ERR_UNSUPPORTED, "pa_prefill: too many query tiles");

    CUtensorMap kv_map, q_map;
    int rc = encode_kv_map(&kv_map, kv_cache, num_blocks, block_size, num_kv_heads);
    if (rc != PA_OK)
        return rc;
    rc = encode_q_map(&q_map, query, total_q, num_q_heads, prm.rows_per_head);
    if (rc != PA_OK)
        return rc;

    const void *fn = dtype == PA_BF16 ? reinterpret_cast<const void *>(&paged_prefill_kernel<true>)
                                      : reinterpret_cast<const void *>(&paged_prefill_kernel<false>);
    // Raise the kernel's shared-memory limit once per device (a call being
    // captured into a CUDA graph then makes no attribute call).
    static std::mutex mu;
    static bool raised[2][64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return set_error(PA_ERR_CUDA, "pa_prefill: cudaGetDevice: %s", cudaGetErrorString(e));
    {
        std::lock_guard<std::mutex> lock(mu);
        bool &done = raised[dtype == PA_BF16][dev & 63];
        if (!done) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess)
                return set_error(PA_ERR_CUDA, "pa_prefill: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            done = dev < 64;
        }
    }
    const dim3 grid((unsigned)(prm.q_tiles * prm.head_tiles), (unsigned)num_kv_heads, (unsigned)num_seqs);
    void *args[] = {&kv_map, &q_map, &prm};
    e = cudaLaunchKernel(fn, grid, dim3(kThreads), args, kSmemBytes, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return set_error(PA_ERR_CUDA, "pa_prefill: launch: %s", cudaGetErrorString(e));
    return PA_OK;
}
