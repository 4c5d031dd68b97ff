// PagedAttention decode for GB300 (sm_103a): kernels and their C ABI.
//
// What is computed follows the PagedAttention pages (vLLM book chapter 4,
// "第4章 PagedAttention：虚拟内存的启示": §4.3.1 pool layout, §4.4 block
// table and slot mapping, §4.5 write-then-read call chain, §4.6 online
// softmax; "PagedAttention: virtual memory for the KV cache": copy-on-write).
// How it is computed is GB300-specific:
//
//  * pa_decode is HBM-bound (a few flops per byte). Each warp streams its own
//    share of 16-token K/V tiles through a private ring of shared-memory
//    stages filled by TMA (cp.async.bulk.tensor, 128-byte swizzle), one
//    mbarrier per stage, with the block-table lookups for the next 32 tiles
//    prefetched into registers. The tile is consumed with ldmatrix and
//    mma.m16n8k16 (fp16/bf16 in, fp32 accumulate): S^T = K Q^T puts the GQA
//    query group on the MMA's N side, P is transposed in registers with
//    movmatrix, and O^T += V^T P^T. The softmax is an fp32 online softmax in
//    base 2.
//  * Work is split "stream-K" style: all 16-token tiles of all (sequence,
//    kv-head, query-tile) segments are laid end to end and every warp of a
//    persistent grid takes an equal contiguous share. A segment inside one
//    warp's share is finished in place; a segment cut by share boundaries
//    leaves one partial (m, l, O) record per piece, and a second kernel,
//    launched with programmatic dependent launch so that it is resident before
//    the first one ends, merges each such segment's pieces in ascending order.
//    The split depends only on the sequence lengths and the grid size, never
//    on physical block ids, so outputs are bit-identical under any
//    permutation of block placement.
//  * reshape_and_cache and copy_blocks are bit copies with 16-byte accesses.
//  * FP8 cache (OCP E4M3 codes with one scale for K and one for V; a reading
//    of the book's "lower-precision KV cache", §4.8): the same pipeline moves
//    half the bytes. Codes are widened to fp16/bf16 in registers (exactly:
//    every E4M3 value is representable in both), so the MMAs, the softmax and
//    the split-K records are those of the 16-bit path; k_scale folds into the
//    score scale and v_scale into the final normalisation. Because a dot
//    product may sum its terms in any order, the head dimension is permuted
//    (the same permutation on Q and K) so that every thread reads its K bytes
//    as whole 16-byte chunks; V's head-dimension rows are permuted too, and
//    the permutation is undone when O is stored.
//  * reshape_and_cache_fp8 quantises with one IEEE fp32 division per element
//    and a saturating round-to-nearest-even conversion.
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

// ---------------------------------------------------------------- device state

__device__ int g_device_error;  // PA_DEVERR_* bits, read and cleared by pa_get_device_error

__device__ __forceinline__ void raise_error(int bit) { atomicOr(&g_device_error, bit); }

// --------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ uint32_t movm_t(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
    return v;
}

// Byte permute: result byte i = byte sel_i of the 8-byte value {b, a}.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Two E4M3 codes (low 16 bits of x: low byte -> low half) to an fp16 pair.
// Exact: every E4M3 value is an fp16 value.
__device__ __forceinline__ uint32_t e4m3x2_lo_to_f16x2(uint32_t x)
{
    uint32_t d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(d)
        : "r"(x));
    return d;
}

// The same for the high 16 bits of x.
__device__ __forceinline__ uint32_t e4m3x2_hi_to_f16x2(uint32_t x)
{
    uint32_t d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, hi;\n\t}"
        : "=r"(d)
        : "r"(x));
    return d;
}

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// ------------------------------------------------------------------- decode

#ifndef PA_DECODE_WARPS
#define PA_DECODE_WARPS 12
#endif
#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 1
#endif
#ifndef PA_DECODE_WARPS_WIDE
#define PA_DECODE_WARPS_WIDE 8
#endif
#ifndef PA_DECODE_STAGES_FP8
#define PA_DECODE_STAGES_FP8 2
#endif

// Warps per CTA, each an independent pipeline: 12 for 8-column query tiles;
// 16-column tiles need ~195 registers per thread, so 8 warps fit an SM.
#ifndef PA_DECODE_WARPS_FP8
#define PA_DECODE_WARPS_FP8 12
#endif
template <int NT, bool FP8 = false>
constexpr int decode_warps()
{
    return NT == 1 ? (FP8 ? PA_DECODE_WARPS_FP8 : PA_DECODE_WARPS) : PA_DECODE_WARPS_WIDE;
}
// TMA ring depth per warp. An FP8 tile is half the bytes of a 16-bit one, so
// the FP8 pipelines keep two in flight to hold the same bytes in flight.
template <bool FP8>
constexpr int decode_stages()
{
    return FP8 ? PA_DECODE_STAGES_FP8 : PA_DECODE_STAGES;
}
constexpr int kTile = 16;       // tokens per tile (the MMA's M)
constexpr int kMaxSeqs = 4096;  // sequences per pa_decode call (prefix lives in smem)

// One pipeline stage: a 16-token tile of one kv head, K rows then V rows.
// 16-bit cache: D/64 TMA boxes [K|V][16 rows][64 elements = 128 B], 128-byte
// swizzle. FP8 cache: one box [K|V][16 rows][D bytes]; D = 128 gives 128-byte
// rows (128-byte swizzle), D = 64 gives 64-byte rows (64-byte swizzle).
template <int D, bool FP8 = false>
struct TileGeo {
    static constexpr int kBoxes = FP8 ? 1 : D / 64;
    static constexpr int kBoxElems = FP8 ? D : 64;          // innermost box extent
    static constexpr int kRowBytes = FP8 ? D : 128;
    static constexpr int kBoxBytes = 2 * kTile * kRowBytes;
    static constexpr int kVOffset = kTile * kRowBytes;      // V rows inside a box
    static constexpr int kStageBytes = kBoxes * kBoxBytes;
};

// Byte offset of 16-byte chunk c of row r inside an FP8 half-tile, after the
// TMA swizzle (128-byte: chunk ^= r mod 8; 64-byte: chunk ^= (r / 2) mod 4).
template <int D>
__device__ __forceinline__ uint32_t fp8_off(int r, int c)
{
    if constexpr (D == 128)
        return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
    else
        return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

struct DecodeParams {
    void *out;
    const uint16_t *query;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    float *warp_records;  // workspace: 2 per warp, the warp's pieces of its first / last segment
    long long *prefix_ws; // workspace: unit prefix over sequences, [num_seqs + 1]
    int4 *tasks;          // workspace: per warp {segment, first owner, first slot, 0} of the
                          // split segment whose last piece it holds; segment -1 if none
    int max_blocks_per_seq;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;            // num_q_heads / num_kv_heads
    int tile_q;           // query heads per query tile (<= 16)
    int qtiles;           // query tiles per kv head
    int num_blocks;
    int block_size;
    int tiles_per_block;  // block_size / 16
    float scale_log2;     // scale * log2(e) (* k_scale for an FP8 cache): scores in base 2
    float v_scale;        // FP8 cache: value of a V code's unit; 1 otherwise
    int kv_stream;        // 1: stream K/V with the L2 evict-first hint (no block shared)
    int lens_early;       // 1: seq_lens may be read before the preceding kernel has finished
    int total_warps;      // grid * warps per CTA
};

template <int D, int NT>
constexpr int record_floats()
{
    return NT * 8 * (D + 2);  // m[GP], l[GP], O[GP][D]; only live query columns are written
}

template <int D, int WARPS, bool FP8>
inline size_t decode_smem_bytes(int num_seqs)
{
    constexpr int kStages = decode_stages<FP8>();
    size_t b = 1024;  // alignment slack for the 1024-byte swizzle atoms
    b += (size_t)WARPS * kStages * TileGeo<D, FP8>::kStageBytes;
    b += (size_t)WARPS * kStages * sizeof(uint64_t);
    b += (size_t)(num_seqs + 1) * sizeof(long long);
    b += (size_t)num_seqs * sizeof(int);
    return b;
}

// The unit sequence: every (sequence, kv head, query tile) segment's 16-token
// tiles laid end to end, sequence-major. prefix[s] is the first unit of
// sequence s; its segments follow one another, ceil(L_s / 16) units each.
struct UnitMap {
    const long long *prefix;  // [num_seqs + 1]
    const int *lens;          // sequence lengths (clamped on read)
    int num_seqs, segs_per_seq, max_len;

    __device__ __forceinline__ int len(int s) const
    {
        const int L = lens[s];
        return L < 0 ? 0 : (L > max_len ? max_len : L);
    }
    __device__ __forceinline__ int seq_of(long long u) const
    {
        int lo = 0, hi = num_seqs;  // prefix[lo] <= u < prefix[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= u)
                lo = mid;
            else
                hi = mid;
        }
        return lo;
    }
    __device__ __forceinline__ int seg_of(long long u) const
    {
        const int s = seq_of(u);
        const int nt = (len(s) + kTile - 1) / kTile;
        return s * segs_per_seq + (int)((u - prefix[s]) / nt);
    }
    __device__ __forceinline__ void bounds(int seg, long long &a, long long &e) const
    {
        const int s = seg / segs_per_seq, segl = seg - (seg / segs_per_seq) * segs_per_seq;
        const int nt = (len(s) + kTile - 1) / kTile;
        a = prefix[s] + (long long)segl * nt;
        e = a + nt;
    }
};

// Equal contiguous shares of N units among K owners: owner k has
// [N k / K, N (k+1) / K); owner_of(u) inverts that.
__device__ __forceinline__ long long share_lo(long long N, long long k, long long K)
{
    return N * k / K;
}
__device__ __forceinline__ int owner_of(long long u, long long N, long long K)
{
    return (int)(((u + 1) * K - 1) / N);
}

// Main decode kernel. Template: head size D, N-tiles of 8 query heads NT,
// element type of Q and the output, FP8 cache or not. One CTA =
// decode_warps<NT>() independent warp pipelines.
template <int D, int NT, bool BF16, bool FP8>
__global__ void __launch_bounds__(decode_warps<NT, FP8>() * 32)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p)
{
    using Geo = TileGeo<D, FP8>;
    constexpr int kWarps = decode_warps<NT, FP8>();
    constexpr int kStages = decode_stages<FP8>();
    constexpr int KS = D / 16;  // k-steps of QK^T and m-tiles of V^T P^T
    constexpr int GP = NT * 8;
    constexpr int STAGE = Geo::kStageBytes;
    constexpr int REC = record_floats<D, NT>();
    // FP8 fragment geometry: each thread reads CPT 16-byte K chunks per row
    // and VB bytes of V per row (see the tile loop).
    constexpr int CPT = D / 64;
    constexpr int VB = D / 8;
    // Operand type of both MMAs: the element type, or fp16 for an FP8 cache
    // (every E4M3 value is an fp16 value; bf16 queries are converted per
    // column, see begin_segment). kPShift scales P by 2^8 in the FP8 case so
    // that fp16 keeps weights down to 2^-32 of the largest.
    constexpr bool MBF16 = BF16 && !FP8;
    constexpr float kPShift = FP8 ? 8.f : 0.f;

    extern __shared__ uint8_t smem_raw[];
    __shared__ long long warp_sums[kWarps];

    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (base - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kWarps * kStages * STAGE);
    long long *prefix = reinterpret_cast<long long *>(bars + kWarps * kStages);
    int *lens = reinterpret_cast<int *>(prefix + p.num_seqs + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.num_seqs;
    const int segs_per_seq = p.num_kv_heads * p.qtiles;
    const int max_len = p.max_blocks_per_seq * p.block_size;

    // Unless the caller vouched that seq_lens is final before the preceding
    // kernel in the stream started, that kernel may still be writing it:
    // wait for it before the first read.
    if (!p.lens_early)
        grid_dependency_wait();

    // 1. Sequence lengths and the exclusive prefix of units (tiles x segments).
    {
        const int per = (S + blockDim.x - 1) / blockDim.x;
        const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
        long long local = 0;
        for (int s = s0; s < s1; ++s) {
            int L = p.seq_lens[s];
            if (L < 0 || L > max_len) {
                raise_error(PA_DEVERR_SEQ_LEN);
                L = L < 0 ? 0 : max_len;
            }
            lens[s] = L;
            local += (long long)((L + kTile - 1) / kTile) * segs_per_seq;
        }
        long long incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o)
                incl += v;
        }
        if (lane == 31)
            warp_sums[warp] = incl;
        __syncthreads();
        long long off = 0;
        for (int w = 0; w < warp; ++w)
            off += warp_sums[w];
        long long run = off + incl - local;
        for (int s = s0; s < s1; ++s) {
            prefix[s] = run;
            run += (long long)((lens[s] + kTile - 1) / kTile) * segs_per_seq;
        }
        if (tid == (int)blockDim.x - 1)
            prefix[S] = off + incl;
    }
    if (lane == 0) {
        for (int st = 0; st < kStages; ++st)
            mbar_init(smem_addr(&bars[warp * kStages + st]), 1);
        fence_barrier_init();
    }
    __syncthreads();

    // Let the reduce kernel start launching; it waits for this grid anyway.
    grid_launch_dependents();
    // Everything above read only the lengths. The pool may still be being
    // written by the preceding kernel (this step's reshape_and_cache): wait
    // for it before any pool read or global write (a no-op if the wait above
    // already ran).
    grid_dependency_wait();

    const long long N = prefix[S];
    if (blockIdx.x == 0)
        for (int s = tid; s <= S; s += blockDim.x)
            p.prefix_ws[s] = prefix[s];
    // Empty sequences get zero output rows (no warp streams them).
    for (int s = blockIdx.x; s < S; s += gridDim.x)
        if (lens[s] == 0)
            for (int i = tid; i < p.num_q_heads * D; i += blockDim.x)
                static_cast<uint16_t *>(p.out)[(long long)s * p.num_q_heads * D + i] = 0;

    // 2. This warp's contiguous share of the unit sequence.
    const int gw = blockIdx.x * kWarps + warp;
    const long long r0 = share_lo(N, gw, p.total_warps);
    const long long r1 = share_lo(N, gw + 1, p.total_warps);
    if (lane == 0)
        p.tasks[gw] = make_int4(-1, 0, 0, 0);
    if (r0 >= r1) {
        // An empty share is a zero-weight piece of whatever segment spans it:
        // mark its first record (m = -inf, l = 0) so merges can skip it.
        float *rec = p.warp_records + 2LL * gw * REC;
        if (lane < p.tile_q) {
            rec[lane] = -INFINITY;
            rec[GP + lane] = 0.f;
        }
        return;
    }

    // Unit u -> physical block, segment id and tv = kv head << 16 | tile
    // index inside its block << 5 | valid tokens (what the TMA issue needs,
    // so that no division runs per tile).
    auto unit_info = [&](long long u, int &phys, int &seg, int &tv) {
        phys = -1;
        seg = -1;
        tv = 0;
        if (u >= r1)
            return;
        int lo = 0, hi = S;  // prefix[lo] <= u < prefix[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= u)
                lo = mid;
            else
                hi = mid;
        }
        const int L = lens[lo];
        const int ntiles = (L + kTile - 1) / kTile;
        const long long local = u - prefix[lo];
        const int segl = (int)(local / ntiles);
        const int tile = (int)(local - (long long)segl * ntiles);
        const int blk = tile / p.tiles_per_block;
        // Not checked here: the load's latency is hidden until issue time.
        phys = __ldg(p.block_tables + (long long)lo * p.max_blocks_per_seq + blk);
        seg = lo * segs_per_seq + segl;
        tv = ((segl / p.qtiles) << 16) | ((tile - blk * p.tiles_per_block) << 5) |
             min(kTile, L - tile * kTile);
    };

    // Register windows of unit info: A covers [wb, wb+32), B covers [wb+32, wb+64).
    long long wb = r0;
    int a_phys, a_seg, a_tv, b_phys, b_seg, b_tv;
    unit_info(wb + lane, a_phys, a_seg, a_tv);
    unit_info(wb + 32 + lane, b_phys, b_seg, b_tv);
    auto fetch = [&](long long v, int &ph, int &sg, int &t) {
        const int idx = (int)(v - wb);
        const bool first = idx < 32;
        const int src = idx & 31;
        ph = __shfl_sync(kFull, first ? a_phys : b_phys, src);
        sg = __shfl_sync(kFull, first ? a_seg : b_seg, src);
        t = __shfl_sync(kFull, first ? a_tv : b_tv, src);
    };

    const uint64_t kv_policy = p.kv_stream ? policy_evict_first() : policy_evict_normal();
    const uint32_t my_stage0 = base + (uint32_t)(warp * kStages * STAGE);
    const uint32_t my_bar0 = smem_addr(&bars[warp * kStages]);
    auto issue = [&](int phys, int seg, int tv, int st) {
        if (lane == 0) {
            if ((unsigned)phys >= (unsigned)p.num_blocks) {
                raise_error(PA_DEVERR_BLOCK_ID);
                phys = p.num_blocks;  // outside the tensor map: TMA fills zeros
            }
            const int h = tv >> 16;
            const int t0 = ((tv >> 5) & 0x7FF) * kTile;
            const uint32_t bar = my_bar0 + st * 8;
            mbar_expect_tx(bar, STAGE);
#pragma unroll
            for (int bx = 0; bx < Geo::kBoxes; ++bx)
                tma_load_5d_hint(my_stage0 + st * STAGE + bx * Geo::kBoxBytes, &kv_map, bar,
                                 bx * Geo::kBoxElems, h, t0, phys, 0, kv_policy);
        }
    };

    long long ip = r0;  // next unit to issue
    for (int st = 0; st < kStages && ip < r1; ++st, ++ip) {
        int ph, sg, t;
        fetch(ip, ph, sg, t);
        issue(ph, sg, t, st);
    }

    const int g = lane >> 2, tig = lane & 3;
    const int k_row = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix rows for K (A of S^T)
    const int k_hi = lane >> 4;
    const int v_row = (lane & 7) + ((lane >> 4) & 1) * 8;  // ldmatrix.trans rows for V (A of O^T)
    const int v_hi = (lane >> 3) & 1;

    float m_run[NT][2], l_run[NT][2], acc[KS][NT][4];
    uint32_t qf[NT][KS][2];
    float xscale[NT][2];  // per-column score scale (bf16 queries on an FP8 cache)
    int cur_seg = -1;

    auto seg_coords = [&](int seg, int &s, int &segl, int &hq0) {
        s = seg / segs_per_seq;
        segl = seg - s * segs_per_seq;
        const int h = segl / p.qtiles, qt = segl - (segl / p.qtiles) * p.qtiles;
        hq0 = h * p.group + qt * 16;
    };

    auto begin_segment = [&](int seg) {
        int s, segl, hq0;
        seg_coords(seg, s, segl, hq0);
        const uint16_t *qbase = p.query + ((long long)s * p.num_q_heads + hq0) * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = nt * 8 + g;
            const bool live = col < p.tile_q;
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(qbase + (long long)col * D);
            if constexpr (FP8) {
                // Permuted k-step kk = 4j + w: dims 16c + 4w + {0..3} of chunk
                // c = CPT tig + j, the same dims the K fragments hold.
                const uint2 *q4 = reinterpret_cast<const uint2 *>(qrow);
                auto q_at = [&](int kk) {
                    return live ? __ldg(q4 + 4 * (CPT * tig + (kk >> 2)) + (kk & 3)) : make_uint2(0u, 0u);
                };
                if constexpr (BF16) {
                    // bf16 column -> fp16 times 2^sh, sh putting the column's
                    // largest element in [2^14, 2^15): exact for every element
                    // within 2^-28 of it (smaller ones round with an error
                    // below 2^-39 of it). The column's score scale takes 2^-sh.
                    int emax = 0;
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk) {
                        const uint2 u = q_at(kk);
                        emax = max(emax, max(max(u.x & 0x7F80, (u.x >> 16) & 0x7F80),
                                             max(u.y & 0x7F80, (u.y >> 16) & 0x7F80)));
                    }
                    emax = max(emax, __shfl_xor_sync(kFull, emax, 1));
                    emax = max(emax, __shfl_xor_sync(kFull, emax, 2));
                    const int sh = min(126, 141 - (emax >> 7));
                    const float s2 = __int_as_float((sh + 127) << 23);
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk) {
                        const uint2 u = q_at(kk);
                        qf[nt][kk][0] = pack2<false>(__uint_as_float(u.x << 16) * s2,
                                                     __uint_as_float(u.x & 0xFFFF0000u) * s2);
                        qf[nt][kk][1] = pack2<false>(__uint_as_float(u.y << 16) * s2,
                                                     __uint_as_float(u.y & 0xFFFF0000u) * s2);
                    }
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int sh_c = __shfl_sync(kFull, sh, (2 * tig + e) << 2);
                        xscale[nt][e] = p.scale_log2 * __int_as_float((127 - sh_c) << 23);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk) {
                        const uint2 u = q_at(kk);
                        qf[nt][kk][0] = u.x;  // dims +0, +1
                        qf[nt][kk][1] = u.y;  // dims +2, +3
                    }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    qf[nt][kk][0] = live ? __ldg(qrow + 8 * kk + tig) : 0u;
                    qf[nt][kk][1] = live ? __ldg(qrow + 8 * kk + 4 + tig) : 0u;
                }
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                m_run[nt][e] = -INFINITY;
                l_run[nt][e] = 0.f;
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    acc[mt][nt][c] = 0.f;
        }
    };

    auto finish_segment = [&](int seg) {
        float lsum[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float v = l_run[nt][e];
                v += __shfl_xor_sync(kFull, v, 4);
                v += __shfl_xor_sync(kFull, v, 8);
                v += __shfl_xor_sync(kFull, v, 16);
                lsum[nt][e] = v;
            }
        int s, segl, hq0;
        seg_coords(seg, s, segl, hq0);
        const int ntiles = (lens[s] + kTile - 1) / kTile;
        const long long seg_start = prefix[s] + (long long)segl * ntiles;
        const long long seg_end = seg_start + ntiles;
        if (seg_start >= r0 && seg_end <= r1) {
            // Whole segment in this warp's share: normalise and store.
            uint16_t *out = static_cast<uint16_t *>(p.out) + ((long long)s * p.num_q_heads + hq0) * D;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = nt * 8 + 2 * tig + e;
                    if (col < p.tile_q) {
                        uint16_t *row = out + (long long)col * D;
                        if constexpr (FP8) {
                            // Rows g / g+8 of m-tile mt are dims VB g + 2mt / + 1.
                            const float inv = p.v_scale / lsum[nt][e];
                            uint32_t *row2 = reinterpret_cast<uint32_t *>(row + VB * g);
#pragma unroll
                            for (int mt = 0; mt < KS; ++mt)
                                row2[mt] = pack2<BF16>(acc[mt][nt][e] * inv, acc[mt][nt][2 + e] * inv);
                        } else {
                            const float inv = 1.f / lsum[nt][e];
#pragma unroll
                            for (int mt = 0; mt < KS; ++mt) {
                                row[16 * mt + g] = to_elem<BF16>(acc[mt][nt][e] * inv);
                                row[16 * mt + g + 8] = to_elem<BF16>(acc[mt][nt][2 + e] * inv);
                            }
                        }
                    }
                }
        } else {
            // A piece of a segment: record (m, l, O) for the reduce kernel.
            // Slot 2w holds the piece of the warp's first segment, 2w+1 its last.
            const long long slot = (seg_start <= r0) ? 2LL * gw : 2LL * gw + 1;
            float *rec = p.warp_records + slot * REC;
            if (lane == 0 && seg_start < r0 && seg_end <= r1) {
                // This warp holds the segment's last piece: post the merge task
                // with the segment's first owner and that owner's record slot.
                const int o_lo = owner_of(seg_start, N, p.total_warps);
                const int first = seg_start == share_lo(N, o_lo, p.total_warps) ? 2 * o_lo : 2 * o_lo + 1;
                p.tasks[gw] = make_int4(seg, o_lo, first, 0);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = nt * 8 + 2 * tig + e;
                    if (col < p.tile_q) {
                        if (g == 0) {
                            rec[col] = m_run[nt][e];
                            rec[GP + col] = lsum[nt][e];
                        }
                        float *ro = rec + 2 * GP + col * D;
                        if constexpr (FP8) {
                            float2 *ro2 = reinterpret_cast<float2 *>(ro + VB * g);
#pragma unroll
                            for (int mt = 0; mt < KS; ++mt)
                                ro2[mt] = make_float2(acc[mt][nt][e] * p.v_scale,
                                                      acc[mt][nt][2 + e] * p.v_scale);
                        } else {
#pragma unroll
                            for (int mt = 0; mt < KS; ++mt) {
                                ro[16 * mt + g] = acc[mt][nt][e];
                                ro[16 * mt + g + 8] = acc[mt][nt][2 + e];
                            }
                        }
                    }
                }
        }
    };

    int st = 0;
    uint32_t phase = 0;
    bool ok = true;
    long long i = r0;
    auto refill = [&]() {
        __syncwarp();
        if (ip < r1) {
            int ph2, sg2, tv2;
            fetch(ip, ph2, sg2, tv2);
            if (lane == 0)
                fence_proxy_async();
            issue(ph2, sg2, tv2, st);
            ++ip;
        }
    };
    for (; i < r1; ++i) {
        if (i - wb >= 32) {
            wb += 32;
            a_phys = b_phys;
            a_seg = b_seg;
            a_tv = b_tv;
            unit_info(wb + 32 + lane, b_phys, b_seg, b_tv);
        }
        int ph, sg, tv;
        fetch(i, ph, sg, tv);
        if (sg != cur_seg) {
            if (cur_seg >= 0)
                finish_segment(cur_seg);
            cur_seg = sg;
            begin_segment(sg);
        }
        if (!mbar_wait(my_bar0 + st * 8, phase)) {
            raise_error(PA_DEVERR_TIMEOUT);
            ok = false;
            break;
        }
        const uint32_t sbuf = my_stage0 + st * STAGE;
        const int valid = tv & 31;
        if (valid < kTile) {
            // Rows past the sequence end hold stale data (possibly NaN): zero the
            // V rows so that p = 0 times them stays 0. K rows are masked below.
            constexpr int CPR = Geo::kRowBytes / 16;  // 16-byte chunks per row
            const int per_box = (kTile - valid) * CPR;
            for (int z = lane; z < per_box * Geo::kBoxes; z += 32) {
                const int bx = z / per_box, rem = z - bx * per_box;
                const int r = valid + rem / CPR, c = rem % CPR;
                sts128_zero(sbuf + bx * Geo::kBoxBytes + Geo::kVOffset + r * Geo::kRowBytes + c * 16);
            }
            fence_proxy_async();
            __syncwarp();
        }

        // S^T[16 tokens][8*NT queries] = K Q^T. All K fragments are loaded
        // first, and the k-steps alternate between two accumulators, so the
        // MMA chain is half as long as the head dimension. V^T fragments do
        // not depend on P: they are loaded up front as well.
        uint32_t kf[KS][4];
        uint32_t vf[KS][4];
        if constexpr (FP8) {
            // K rows g and g+8, chunks c = CPT tig + j, widened in registers.
            // Word w of chunk j holds the dims of permuted k-step 4j + w.
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                const int c = CPT * tig + j;
                const uint4 r0 = lds128(sbuf + fp8_off<D>(g, c));
                const uint4 r1 = lds128(sbuf + fp8_off<D>(g + 8, c));
                const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w};
                const uint32_t w1[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const int kk = 4 * j + w;
                    kf[kk][0] = e4m3x2_lo_to_f16x2(w0[w]);  // dims +0, +1
                    kf[kk][1] = e4m3x2_lo_to_f16x2(w1[w]);
                    kf[kk][2] = e4m3x2_hi_to_f16x2(w0[w]);  // dims +2, +3
                    kf[kk][3] = e4m3x2_hi_to_f16x2(w1[w]);
                }
            }
            // V^T: this thread's dims VB g .. VB g + VB - 1 of tokens 2tig,
            // 2tig+1, 2tig+8, 2tig+9; m-tile mt takes dims VB g + 2mt (row g)
            // and VB g + 2mt + 1 (row g+8), paired across tokens with prmt.
            const uint32_t vbase = sbuf + Geo::kVOffset;
            uint32_t vw[4][VB / 4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int r = 2 * tig + (t & 1) + (t >> 1) * 8;
                if constexpr (D == 128) {
                    const uint4 x = lds128(vbase + fp8_off<D>(r, g));
                    vw[t][0] = x.x;
                    vw[t][1] = x.y;
                    vw[t][2] = x.z;
                    vw[t][3] = x.w;
                } else {
                    const uint2 x = lds64(vbase + fp8_off<D>(r, g >> 1) + ((g & 1) << 3));
                    vw[t][0] = x.x;
                    vw[t][1] = x.y;
                }
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const int wi = mt >> 1;
                // {t.d, t'.d, t.d+1, t'.d+1}: low pair -> row g, high -> row g+8.
                const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
                const uint32_t x01 = prmt(vw[0][wi], vw[1][wi], sel);
                const uint32_t x23 = prmt(vw[2][wi], vw[3][wi], sel);
                vf[mt][0] = e4m3x2_lo_to_f16x2(x01);
                vf[mt][1] = e4m3x2_hi_to_f16x2(x01);
                vf[mt][2] = e4m3x2_lo_to_f16x2(x23);
                vf[mt][3] = e4m3x2_hi_to_f16x2(x23);
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                const int cg = 2 * kk + k_hi;
                ldsm_x4(sbuf + (cg >> 3) * Geo::kBoxBytes + k_row * 128 +
                            (((cg & 7) ^ (k_row & 7)) << 4),
                        kf[kk][0], kf[kk][1], kf[kk][2], kf[kk][3]);
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const int cg = 2 * mt + v_hi;
                ldsm_x4_t(sbuf + 2048 + (cg >> 3) * Geo::kBoxBytes + v_row * 128 +
                              (((cg & 7) ^ (v_row & 7)) << 4),
                          vf[mt][0], vf[mt][1], vf[mt][2], vf[mt][3]);
            }
        }

        float sc[NT][4], sc2[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                sc[nt][c] = sc2[nt][c] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; kk += 2)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                mma16816<MBF16>(sc[nt], kf[kk][0], kf[kk][1], kf[kk][2], kf[kk][3], qf[nt][kk][0],
                                qf[nt][kk][1]);
                mma16816<MBF16>(sc2[nt], kf[kk + 1][0], kf[kk + 1][1], kf[kk + 1][2], kf[kk + 1][3],
                                qf[nt][kk + 1][0], qf[nt][kk + 1][1]);
            }
        // Every fragment of this tile is now in registers: hand the stage back
        // to the TMA right away, so the ring stays full while the math runs.
        refill();

        // Online softmax (base 2) per query column. P is rounded to the
        // element type; with an FP8 cache it is rounded to fp16 (V is widened
        // to fp16) and carries a factor 2^8 (P <= 256), which l and O share.
        const bool tok0 = g < valid, tok1 = g + 8 < valid;
        float alpha[NT][2];
        bool grew = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float xs = (FP8 && BF16) ? xscale[nt][e] : p.scale_log2;
                const float x0 = tok0 ? (sc[nt][e] + sc2[nt][e]) * xs : -INFINITY;
                const float x1 = tok1 ? (sc[nt][2 + e] + sc2[nt][2 + e]) * xs : -INFINITY;
                float mx = fmaxf(x0, x1);
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
                const float m_new = fmaxf(m_run[nt][e], mx);
                grew |= m_new != m_run[nt][e];
                alpha[nt][e] = ex2(m_run[nt][e] - m_new);
                m_run[nt][e] = m_new;
                const float mref = m_new - kPShift;
                sc[nt][e] = ex2(x0 - mref);
                sc[nt][2 + e] = ex2(x1 - mref);
            }
        // Rescale l and O only when some column's maximum grew (alpha != 1):
        // after the first tiles of a segment that is rare.
        if (__any_sync(kFull, grew)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    l_run[nt][e] *= alpha[nt][e];
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        acc[mt][nt][e] *= alpha[nt][e];
                        acc[mt][nt][2 + e] *= alpha[nt][e];
                    }
                }
        }
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint32_t r0p = pack2<MBF16>(sc[nt][0], sc[nt][1]);  // token g,   columns 2tig, 2tig+1
            const uint32_t r1p = pack2<MBF16>(sc[nt][2], sc[nt][3]);  // token g+8
            const float2 f0 = unpack2<MBF16>(r0p), f1 = unpack2<MBF16>(r1p);
            l_run[nt][0] += f0.x + f1.x;
            l_run[nt][1] += f0.y + f1.y;
            pb[nt][0] = movm_t(r0p);  // P^T fragments as the B operand
            pb[nt][1] = movm_t(r1p);
        }

        // O^T[D][8*NT] += V^T P^T
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma16816<MBF16>(acc[mt][nt], vf[mt][0], vf[mt][1], vf[mt][2], vf[mt][3], pb[nt][0],
                                pb[nt][1]);

        if (++st == kStages) {
            st = 0;
            phase ^= 1;
        }
    }
    if (ok) {
        if (cur_seg >= 0)
            finish_segment(cur_seg);
    } else {
        // Give the copies still in flight into this warp's stages a bounded
        // chance to land before the CTA's shared memory goes away.
        for (long long u = i; u < ip; ++u) {
            const int rel = (int)(u - r0);
            mbar_wait(my_bar0 + (rel % kStages) * 8, (uint32_t)((rel / kStages) & 1));
        }
    }
}

// Running merge state of one warp: for every live query column c, the
// maximum M[c], the normaliser l[c] and the rows d = lane + 32 k of O.
template <int D, int NT>
struct MergeState {
    static constexpr int GP = NT * 8, KD = D / 32;
    float M[GP], l[GP], acc[GP][KD];
    __device__ void clear()
    {
#pragma unroll
        for (int c = 0; c < GP; ++c) {
            M[c] = -INFINITY;
            l[c] = 0.f;
#pragma unroll
            for (int k = 0; k < KD; ++k)
                acc[c][k] = 0.f;
        }
    }
};

// Fold the pieces o = o_first, o_first + ostep, ... <= o_hi into the state.
// Piece o's record is slot first_slot when o == o_lo, else 2o. PPR pieces
// are loaded per round (m, l and the O rows together) and folded with the
// online-softmax rule; a piece with m = -inf (an empty share) weighs 0.
template <int D, int NT>
__device__ void fold_pieces(const float *recs, int o_first, int ostep, int o_hi, int o_lo,
                            int first_slot, int tq, MergeState<D, NT> &st)
{
    constexpr int GP = NT * 8, KD = D / 32, REC = record_floats<D, NT>();
    constexpr int PPR = NT == 1 ? 2 : 1;
    const int lane = threadIdx.x & 31;
    for (int o0 = o_first; o0 <= o_hi; o0 += PPR * ostep) {
        float mp[PPR][GP], lp[PPR][GP], x[PPR][GP][KD];
#pragma unroll
        for (int j = 0; j < PPR; ++j) {
            const int o = o0 + j * ostep;
            const bool ok = o <= o_hi;
            const float *r = recs + (long long)(o == o_lo ? first_slot : 2 * o) * REC;
#pragma unroll
            for (int c = 0; c < GP; ++c) {
                const bool live = ok && c < tq;
                mp[j][c] = live ? __ldcg(r + c) : -INFINITY;
                lp[j][c] = live ? __ldcg(r + GP + c) : 0.f;
#pragma unroll
                for (int k = 0; k < KD; ++k)
                    x[j][c][k] = live ? __ldcg(r + 2 * GP + c * D + lane + 32 * k) : 0.f;
            }
        }
        // A marked empty share (m = -inf) has no O rows: never read them.
#pragma unroll
        for (int j = 0; j < PPR; ++j)
#pragma unroll
            for (int c = 0; c < GP; ++c)
                if (mp[j][c] == -INFINITY) {
                    lp[j][c] = 0.f;
#pragma unroll
                    for (int k = 0; k < KD; ++k)
                        x[j][c][k] = 0.f;
                }
#pragma unroll
        for (int c = 0; c < GP; ++c) {
            float mb = st.M[c];
#pragma unroll
            for (int j = 0; j < PPR; ++j)
                mb = fmaxf(mb, mp[j][c]);
            if (mb == -INFINITY)
                continue;  // nothing valid in this column yet
            const float scale = ex2(st.M[c] - mb);  // 0 on the first valid piece
            float f[PPR];
#pragma unroll
            for (int j = 0; j < PPR; ++j)
                f[j] = mp[j][c] == -INFINITY ? 0.f : ex2(mp[j][c] - mb);
            float lv = st.l[c] * scale;
#pragma unroll
            for (int j = 0; j < PPR; ++j)
                lv += f[j] * lp[j][c];
            st.l[c] = lv;
#pragma unroll
            for (int k = 0; k < KD; ++k) {
                float v = st.acc[c][k] * scale;
#pragma unroll
                for (int j = 0; j < PPR; ++j)
                    v += f[j] * x[j][c][k];
                st.acc[c][k] = v;
            }
            st.M[c] = mb;
        }
    }
}

constexpr int kSmallTask = 6;    // pieces a single warp merges on its own
constexpr int kReduceWarps = 4;  // warps per reduce CTA

template <int D, int NT>
constexpr size_t reduce_smem_bytes()
{
    return (size_t)kReduceWarps * (2 * NT * 8 + D * NT * 8) * sizeof(float);  // per warp: M, l, O
}

// Finish the segments cut by warp-share boundaries. Warp j of reduce CTA r
// serves main-grid warp
// r * kReduceWarps + j: if that warp holds the last piece of a split segment,
// the segment's pieces (one record per main-grid warp, ascending) are merged
// with the online-softmax rule m = max m_p, l = sum l_p 2^(m_p - m),
// O = sum O_p 2^(m_p - m). A task with few pieces is merged by its warp; a
// task with many pieces by the whole CTA, pieces split across the warps and
// the warps' states combined in shared memory. Every merge runs in a fixed
// order, so results do not depend on timing.
template <int D, int NT, bool BF16>
__global__ void __launch_bounds__(kReduceWarps * 32) paged_decode_reduce_kernel(const DecodeParams p)
{
    constexpr int GP = NT * 8, KD = D / 32, PART = 2 * GP + GP * D;
    extern __shared__ float s_part[];  // [kReduceWarps][M GP | l GP | O GP x D]
    __shared__ int4 s_task[kReduceWarps];

    grid_dependency_wait();  // the main grid's records and tasks are complete
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w = blockIdx.x * kReduceWarps + warp;
    const int tq = p.tile_q;
    const int segs_per_seq = p.num_kv_heads * p.qtiles;
    uint16_t *out_base = static_cast<uint16_t *>(p.out);
    auto out_rows = [&](int seg) {
        const int s = seg / segs_per_seq, segl = seg - (seg / segs_per_seq) * segs_per_seq;
        const int h = segl / p.qtiles, qt = segl - (segl / p.qtiles) * p.qtiles;
        return out_base + ((long long)s * p.num_q_heads + h * p.group + qt * 16) * D;
    };
    auto store = [&](uint16_t *out, const MergeState<D, NT> &st) {
#pragma unroll
        for (int c = 0; c < GP; ++c)
            if (c < tq) {
                const float inv = 1.f / st.l[c];
#pragma unroll
                for (int k = 0; k < KD; ++k)
                    out[(long long)c * D + lane + 32 * k] = to_elem<BF16>(st.acc[c][k] * inv);
            }
    };

    const int4 task = w < p.total_warps ? p.tasks[w] : make_int4(-1, 0, 0, 0);
    const bool small = task.x >= 0 && w - task.y + 1 <= kSmallTask;
    if (lane == 0)
        s_task[warp] = (task.x >= 0 && !small) ? task : make_int4(-1, 0, 0, 0);
    if (small) {
        MergeState<D, NT> st;
        st.clear();
        fold_pieces<D, NT>(p.warp_records, task.y, 1, w, task.y, task.z, tq, st);
        store(out_rows(task.x), st);
    }
    __syncthreads();
    // Tasks with many pieces: the whole CTA, pieces split across warps.
    for (int j = 0; j < kReduceWarps; ++j) {
        const int4 t = s_task[j];
        if (t.x < 0)
            continue;
        const int last = blockIdx.x * kReduceWarps + j;
        MergeState<D, NT> st;
        st.clear();
        fold_pieces<D, NT>(p.warp_records, t.y + warp, kReduceWarps, last, t.y, t.z, tq, st);
        float *mine = s_part + warp * PART;
#pragma unroll
        for (int c = 0; c < GP; ++c) {
            if (lane == 0) {
                mine[c] = st.M[c];
                mine[GP + c] = st.l[c];
            }
#pragma unroll
            for (int k = 0; k < KD; ++k)
                mine[2 * GP + c * D + lane + 32 * k] = st.acc[c][k];
        }
        __syncthreads();
        // Combine the warps' states (fixed order), elements across the CTA.
        uint16_t *out = out_rows(t.x);
        for (int e = threadIdx.x; e < tq * D; e += kReduceWarps * 32) {
            const int c = e / D, d = e - (e / D) * D;
            float Mx = -INFINITY;
            for (int v = 0; v < kReduceWarps; ++v)
                Mx = fmaxf(Mx, s_part[v * PART + c]);
            float lt = 0.f, ot = 0.f;
            for (int v = 0; v < kReduceWarps; ++v) {
                const float *pv = s_part + v * PART;
                const float f = pv[c] == -INFINITY ? 0.f : ex2(pv[c] - Mx);  // warp had no pieces
                lt += f * pv[GP + c];
                ot += f * pv[2 * GP + c * D + d];
            }
            out[(long long)c * D + d] = to_elem<BF16>(ot / lt);
        }
        __syncthreads();
    }
}

// ------------------------------------------------------- reshape and copy

// One CTA per token: the token's K row [num_kv_heads][head_size] and V row
// are contiguous both in the input and in the pool. Each thread moves
// kReshapeVecs 16-byte elements of each, all loads issued before the stores
// (so that many bytes are in flight); the block is sized to the row.
constexpr int kReshapeVecs = 4;
constexpr int kReshapeMaxThreads = 256;

__global__ void __launch_bounds__(kReshapeMaxThreads)
    reshape_and_cache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                             uint4 *__restrict__ kv, const int32_t *__restrict__ slots,
                             int row_vecs, long long num_slots, long long half_vecs)
{
    grid_launch_dependents();  // the decode that follows may start its prologue
    const int t = blockIdx.x;
    const long long slot = slots[t];
    if (slot < 0)
        return;
    if (slot >= num_slots) {
        if (threadIdx.x == 0)
            raise_error(PA_DEVERR_SLOT);
        return;
    }
    const uint4 *ksrc = key + (long long)t * row_vecs, *vsrc = value + (long long)t * row_vecs;
    uint4 *kdst = kv + slot * row_vecs, *vdst = kv + half_vecs + slot * row_vecs;
    for (int base = threadIdx.x; base < row_vecs; base += blockDim.x * kReshapeVecs) {
        uint4 k[kReshapeVecs], v[kReshapeVecs];
#pragma unroll
        for (int u = 0; u < kReshapeVecs; ++u) {
            const int i = base + u * blockDim.x;
            if (i < row_vecs) {
                k[u] = __ldg(ksrc + i);
                v[u] = __ldg(vsrc + i);
            }
        }
#pragma unroll
        for (int u = 0; u < kReshapeVecs; ++u) {
            const int i = base + u * blockDim.x;
            if (i < row_vecs) {
                kdst[i] = k[u];
                vdst[i] = v[u];
            }
        }
    }
}

// Two fp32 values to E4M3 codes (saturating, nearest-even); `lo` goes to the
// low byte of the result.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi)
{
    uint32_t d;
    asm("{\n\t.reg .b16 r;\n\tcvt.rn.satfinite.e4m3x2.f32 r, %1, %2;\n\t"
        "cvt.u32.u16 %0, r;\n\t}"
        : "=r"(d)
        : "f"(hi), "f"(lo));
    return d;
}

// Eight 16-bit elements to eight codes of element / scale (one IEEE fp32
// division each).
template <bool BF16>
__device__ __forceinline__ uint2 quantize8(const uint4 x, float scale)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = unpack2<BF16>(w[i]);
        c[i] = f32x2_to_e4m3x2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
    }
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// FP8 write path, grid (token, chunk of kReshapeThreads vectors of the row):
// each thread quantises 8 elements of the token's K row and 8 of its V row
// (16 bytes in, 8 out).
constexpr int kReshapeThreads = 256;
template <bool BF16>
__global__ void __launch_bounds__(kReshapeThreads)
    reshape_and_cache_fp8_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                                 uint2 *__restrict__ kv, const int32_t *__restrict__ slots,
                                 int row_vecs, long long num_slots, long long half_vecs,
                                 float k_scale, float v_scale)
{
    grid_launch_dependents();
    const int t = blockIdx.x;
    const int i = blockIdx.y * kReshapeThreads + threadIdx.x;
    const long long slot = slots[t];
    if (slot < 0)
        return;
    if (slot >= num_slots) {
        if (threadIdx.x == 0 && blockIdx.y == 0)
            raise_error(PA_DEVERR_SLOT);
        return;
    }
    if (i < row_vecs) {
        const uint4 k = __ldg(key + (long long)t * row_vecs + i);
        const uint4 v = __ldg(value + (long long)t * row_vecs + i);
        kv[slot * row_vecs + i] = quantize8<BF16>(k, k_scale);
        kv[half_vecs + slot * row_vecs + i] = quantize8<BF16>(v, v_scale);
    }
}

constexpr int kMaxLayers = 512;
struct LayerPtrs {
    uint4 *p[kMaxLayers];
};

// One CTA per (pair, layer): validate the pair against every other pair,
// then copy the K block and the V block with 16-byte accesses.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(const __grid_constant__ LayerPtrs layers, const int32_t *__restrict__ pairs,
                       int num_pairs, int num_blocks, long long block_vecs, long long half_vecs)
{
    const int i = blockIdx.x, layer = blockIdx.y;
    const int src = pairs[2 * i], dst = pairs[2 * i + 1];
    int clash = ((unsigned)src >= (unsigned)num_blocks || (unsigned)dst >= (unsigned)num_blocks);
    for (int j = threadIdx.x; j < num_pairs; j += blockDim.x) {
        const int sj = pairs[2 * j], dj = pairs[2 * j + 1];
        if (sj == dst || (j != i && dj == dst))
            clash = 1;
    }
    if (__syncthreads_or(clash)) {
        if (threadIdx.x == 0 && layer == 0)
            raise_error(PA_DEVERR_PAIR);
        return;
    }
    uint4 *pool = layers.p[layer];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const uint4 *s = pool + c * half_vecs + (long long)src * block_vecs;
        uint4 *d = pool + c * half_vecs + (long long)dst * block_vecs;
        long long k = threadIdx.x;
        for (; k + 3 * blockDim.x < block_vecs; k += 4 * blockDim.x) {
            const uint4 x0 = s[k], x1 = s[k + blockDim.x], x2 = s[k + 2 * blockDim.x],
                        x3 = s[k + 3 * blockDim.x];
            d[k] = x0;
            d[k + blockDim.x] = x1;
            d[k + 2 * blockDim.x] = x2;
            d[k + 3 * blockDim.x] = x3;
        }
        for (; k < block_vecs; k += blockDim.x)
            d[k] = s[k];
    }
}

// ================================================================ host side

namespace {

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_fail(cudaError_t e, const char *what)
{
    return set_error(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Rank-5 view of the pool, innermost first: (head_size, kv_heads, block
// slots, blocks, K|V). A box is 64 elements x 1 head x 16 slots x 1 block x
// {K, V}: one 16-token tile of one head, K and V together, 128-byte swizzled.
struct MapKey {
    const void *ptr;
    int d, h, b, nb, dev, fp8;
};

// FP8 pools use 1-byte elements and a box of the whole head (D bytes) with
// the swizzle that matches that row length.
int encode_kv_map(CUtensorMap *map, const void *kv, int num_blocks, int block_size,
                  int num_kv_heads, int head_size, int device, bool fp8)
{
    static std::mutex mu;
    // One entry per (pool, shape, device): enough for every layer of a model
    // (each layer has its own pool), so a model step re-encodes nothing.
    constexpr int kMapCache = 128;
    static MapKey keys[kMapCache];
    static CUtensorMap maps[kMapCache];
    static int used = 0, next = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i) {
        const MapKey &k = keys[i];
        if (k.ptr == kv && k.d == head_size && k.h == num_kv_heads && k.b == block_size &&
            k.nb == num_blocks && k.dev == device && k.fp8 == (int)fp8) {
            *map = maps[i];
            return PA_OK;
        }
    }
    auto enc = tensor_map_encoder();
    if (!enc)
        return set_error(PA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t e = fp8 ? 1 : 2;  // bytes per element
    cuuint64_t dims[5] = {(cuuint64_t)head_size, (cuuint64_t)num_kv_heads, (cuuint64_t)block_size,
                          (cuuint64_t)num_blocks, 2};
    cuuint64_t strides[4] = {head_size * e, (cuuint64_t)num_kv_heads * head_size * e,
                             (cuuint64_t)block_size * num_kv_heads * head_size * e,
                             (cuuint64_t)num_blocks * block_size * num_kv_heads * head_size * e};
    cuuint32_t box[5] = {fp8 ? (cuuint32_t)head_size : 64u, 1, (cuuint32_t)kTile, 1, 2};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUtensorMapSwizzle swz =
        (fp8 && head_size == 64) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    // A 16-bit row of one head is 256 bytes (fetched as two 128-byte boxes):
    // promote to 256-byte L2 lines. An FP8 row is at most 128 bytes, and a
    // 256-byte promotion would also pull the next head's row from DRAM.
    const CUtensorMapL2promotion promo =
        fp8 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    CUtensorMap m;
    CUresult r = enc(&m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 5,
                     const_cast<void *>(kv), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swz, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    const int slot = used < kMapCache ? used++ : (next++ % kMapCache);
    keys[slot] = MapKey{kv, head_size, num_kv_heads, block_size, num_blocks, device, (int)fp8};
    maps[slot] = m;
    *map = m;
    return PA_OK;
}

// Launch with programmatic stream serialisation: the kernel may begin while
// the previous kernel in the stream finishes; it calls griddepcontrol.wait
// before touching anything that kernel writes.
cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, void **args, size_t smem,
                       cudaStream_t stream)
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

// Shape and kernel choice for one pa_decode call.
struct DecodePlan {
    int nt = 1;       // 8-query N-tiles
    int tile_q = 1;
    int qtiles = 1;
    int grid = 0;     // CTAs
    int warps = 0;    // warps per CTA
    int total_warps = 0;
    size_t smem = 0;
    size_t prefix_bytes = 0;
    size_t task_bytes = 0;  // one int4 task per warp
    size_t warp_record_bytes = 0;
    const void *main_fn = nullptr;
    const void *reduce_fn = nullptr;
    size_t reduce_smem = 0;
    size_t total() const { return prefix_bytes + task_bytes + warp_record_bytes; }
};

template <int D, int NT, bool BF16, bool FP8>
void pick_kernels(DecodePlan &pl, int num_seqs)
{
    pl.main_fn = reinterpret_cast<const void *>(&paged_decode_kernel<D, NT, BF16, FP8>);
    pl.warps = decode_warps<NT, FP8>();
    pl.reduce_fn = reinterpret_cast<const void *>(&paged_decode_reduce_kernel<D, NT, BF16>);
    pl.reduce_smem = reduce_smem_bytes<D, NT>();
    pl.smem = decode_smem_bytes<D, decode_warps<NT, FP8>(), FP8>(num_seqs);
}

template <int D, int NT>
void pick_kernels(DecodePlan &pl, int num_seqs, bool bf, bool fp8)
{
    if (fp8)
        bf ? pick_kernels<D, NT, true, true>(pl, num_seqs) : pick_kernels<D, NT, false, true>(pl, num_seqs);
    else
        bf ? pick_kernels<D, NT, true, false>(pl, num_seqs) : pick_kernels<D, NT, false, false>(pl, num_seqs);
}

int validate_decode_shape(int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
                          int block_size, int dtype)
{
    if (num_seqs < 0 || num_seqs > kMaxSeqs)
        return set_error(PA_ERR_INVALID_ARG, "pa_decode: num_seqs %d outside [0, %d]", num_seqs, kMaxSeqs);
    if (dtype != PA_F16 && dtype != PA_BF16)
        return set_error(PA_ERR_UNSUPPORTED, "pa_decode: dtype %d (want PA_F16 or PA_BF16)", dtype);
    if (head_size != 64 && head_size != 128)
        return set_error(PA_ERR_UNSUPPORTED, "pa_decode: head_size %d (built: 64, 128)", head_size);
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return set_error(PA_ERR_INVALID_ARG, "pa_decode: num_q_heads %d must be a positive multiple of num_kv_heads %d",
                         num_q_heads, num_kv_heads);
    const int group = num_q_heads / num_kv_heads;
    if (group > 16 && group % 16 != 0)
        return set_error(PA_ERR_UNSUPPORTED, "pa_decode: query group %d (want <= 16 or a multiple of 16)", group);
    if (block_size < kTile || block_size % kTile != 0)
        return set_error(PA_ERR_INVALID_ARG, "pa_decode: block_size %d must be a positive multiple of 16", block_size);
    if (block_size > 2048 * kTile || num_kv_heads > 65535)
        return set_error(PA_ERR_UNSUPPORTED, "pa_decode: block_size %d (max %d) or num_kv_heads %d (max 65535)",
                         block_size, 2048 * kTile, num_kv_heads);
    return PA_OK;
}

// Per (kernel, device): the dynamic shared memory the kernel may use (raised
// on demand) and the occupancy at the last size asked for, so that a call
// makes no attribute or occupancy query once its shape has been seen (and a
// call being captured into a CUDA graph makes none).
cudaError_t kernel_setup(const void *fn, int dev, size_t smem, int threads, int *occ)
{
    struct Entry {
        const void *fn;
        int dev;
        size_t allowed, occ_smem;
        int occ;
    };
    constexpr int kEntries = 64;
    static Entry table[kEntries];
    static int used = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    Entry *e = nullptr;
    for (int i = 0; i < used; ++i)
        if (table[i].fn == fn && table[i].dev == dev)
            e = &table[i];
    if (!e) {
        e = &table[used < kEntries ? used++ : kEntries - 1];
        *e = Entry{fn, dev, 0, (size_t)-1, 0};
    }
    if (smem > e->allowed) {
        cudaError_t r = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (r != cudaSuccess)
            return r;
        e->allowed = smem;
    }
    if (occ) {
        if (e->occ_smem != smem) {
            cudaError_t r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&e->occ, fn, threads, smem);
            if (r != cudaSuccess)
                return r;
            e->occ_smem = smem;
        }
        *occ = e->occ;
    }
    return cudaSuccess;
}

int make_plan(DecodePlan &pl, int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
              int dtype, bool fp8)
{
    const int group = num_q_heads / num_kv_heads;
    pl.tile_q = group <= 16 ? group : 16;
    pl.qtiles = group <= 16 ? 1 : group / 16;
    pl.nt = pl.tile_q <= 8 ? 1 : 2;
    const bool bf = dtype == PA_BF16;
    if (head_size == 64)
        pl.nt == 1 ? pick_kernels<64, 1>(pl, num_seqs, bf, fp8) : pick_kernels<64, 2>(pl, num_seqs, bf, fp8);
    else
        pl.nt == 1 ? pick_kernels<128, 1>(pl, num_seqs, bf, fp8) : pick_kernels<128, 2>(pl, num_seqs, bf, fp8);
    int dev = 0, sms = 0, occ = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    e = kernel_setup(pl.main_fn, dev, pl.smem, pl.warps * 32, &occ);
    if (e != cudaSuccess)
        return cuda_fail(e, "pa_decode: kernel attributes / occupancy");
    e = kernel_setup(pl.reduce_fn, dev, pl.reduce_smem, kReduceWarps * 32, nullptr);
    if (e != cudaSuccess)
        return cuda_fail(e, "pa_decode: reduce kernel attributes");
    if (occ < 1)
        return set_error(PA_ERR_UNSUPPORTED, "pa_decode: kernel does not fit on an SM (smem %zu)", pl.smem);
    pl.grid = sms * occ;
    pl.total_warps = pl.grid * pl.warps;
    const size_t rec = (size_t)pl.nt * 8 * (head_size + 2) * sizeof(float);
    pl.prefix_bytes = ((size_t)(num_seqs + 1) * sizeof(long long) + 255) / 256 * 256;
    pl.task_bytes = ((size_t)pl.total_warps * sizeof(int4) + 255) / 256 * 256;
    pl.warp_record_bytes = 2 * (size_t)pl.total_warps * rec;
    return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

namespace {

int workspace_size_impl(const char *fn, int num_seqs, int num_q_heads, int num_kv_heads,
                        int head_size, int block_size, int dtype, bool fp8, size_t *bytes)
{
    if (!bytes)
        return set_error(PA_ERR_INVALID_ARG, "%s: bytes is null", fn);
    int rc = validate_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_size, block_size, dtype);
    if (rc != PA_OK)
        return rc;
    DecodePlan pl;
    rc = make_plan(pl, num_seqs, num_q_heads, num_kv_heads, head_size, dtype, fp8);
    if (rc != PA_OK)
        return rc;
    *bytes = pl.total();
    return PA_OK;
}

int decode_impl(const char *fn, void *out, const void *query, const void *kv_cache,
                const int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_lens,
                int num_seqs, float scale, int num_q_heads, int num_kv_heads, int head_size,
                int num_blocks, int block_size, int dtype, bool fp8, float k_scale, float v_scale,
                void *workspace, size_t workspace_bytes, unsigned flags, pa_stream_t stream)
{
    int rc = validate_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_size, block_size, dtype);
    if (rc != PA_OK)
        return rc;
    if (fp8 && !(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
        return set_error(PA_ERR_INVALID_ARG, "%s: k_scale and v_scale must be finite and > 0", fn);
    if (num_seqs == 0)
        return PA_OK;
    if (!out || !query || !kv_cache || !block_tables || !seq_lens || !workspace)
        return set_error(PA_ERR_INVALID_ARG, "%s: null pointer argument", fn);
    if (num_blocks <= 0 || max_blocks_per_seq <= 0)
        return set_error(PA_ERR_INVALID_ARG, "%s: num_blocks and max_blocks_per_seq must be > 0", fn);
    if ((long long)max_blocks_per_seq * block_size > (1LL << 30))
        return set_error(PA_ERR_INVALID_ARG, "%s: max_blocks_per_seq * block_size too large", fn);
    if (!std::isfinite(scale))
        return set_error(PA_ERR_INVALID_ARG, "%s: scale is not finite", fn);
    if (flags & ~(PA_DECODE_SHARED_BLOCKS | PA_DECODE_LENS_READY))
        return set_error(PA_ERR_INVALID_ARG, "%s: unknown flags 0x%x", fn, flags);
    if (!aligned(kv_cache, 16) || !aligned(query, 16) || !aligned(out, 16) ||
        !aligned(workspace, 256) || !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return set_error(PA_ERR_INVALID_ARG, "%s: misaligned pointer (pool/query/out 16 B, workspace 256 B)", fn);
    DecodePlan pl;
    rc = make_plan(pl, num_seqs, num_q_heads, num_kv_heads, head_size, dtype, fp8);
    if (rc != PA_OK)
        return rc;
    if (workspace_bytes < pl.total())
        return set_error(PA_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu needed", fn, workspace_bytes,
                         pl.total());
    int dev = 0;
    cudaGetDevice(&dev);
    CUtensorMap map;
    rc = encode_kv_map(&map, kv_cache, num_blocks, block_size, num_kv_heads, head_size, dev, fp8);
    if (rc != PA_OK)
        return rc;

    DecodeParams prm;
    prm.out = out;
    prm.query = static_cast<const uint16_t *>(query);
    prm.block_tables = block_tables;
    prm.seq_lens = seq_lens;
    char *ws = static_cast<char *>(workspace);
    prm.prefix_ws = reinterpret_cast<long long *>(ws);
    prm.tasks = reinterpret_cast<int4 *>(ws + pl.prefix_bytes);
    prm.warp_records = reinterpret_cast<float *>(ws + pl.prefix_bytes + pl.task_bytes);
    prm.max_blocks_per_seq = max_blocks_per_seq;
    prm.num_seqs = num_seqs;
    prm.num_q_heads = num_q_heads;
    prm.num_kv_heads = num_kv_heads;
    prm.group = num_q_heads / num_kv_heads;
    prm.tile_q = pl.tile_q;
    prm.qtiles = pl.qtiles;
    prm.num_blocks = num_blocks;
    prm.block_size = block_size;
    prm.tiles_per_block = block_size / kTile;
    prm.scale_log2 = (fp8 ? scale * k_scale : scale) * 1.4426950408889634f;
    prm.v_scale = fp8 ? v_scale : 1.f;
    prm.kv_stream = (flags & PA_DECODE_SHARED_BLOCKS) ? 0 : 1;
    prm.lens_early = (flags & PA_DECODE_LENS_READY) ? 1 : 0;
    prm.total_warps = pl.total_warps;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *args[] = {&map, &prm};
    cudaError_t e = launch_pdl(pl.main_fn, dim3(pl.grid), dim3(pl.warps * 32), args, pl.smem, s);
    if (e != cudaSuccess)
        return set_error(PA_ERR_CUDA, "%s: main kernel launch: %s", fn, cudaGetErrorString(e));
    void *red_args[] = {&prm};
    e = launch_pdl(pl.reduce_fn, dim3((pl.total_warps + kReduceWarps - 1) / kReduceWarps),
                   dim3(kReduceWarps * 32), red_args, pl.reduce_smem, s);
    if (e != cudaSuccess)
        return set_error(PA_ERR_CUDA, "%s: reduce kernel launch: %s", fn, cudaGetErrorString(e));
    return PA_OK;
}

// Checks shared by both write paths; *row_vecs = 8-element groups per row.
int validate_reshape(const char *fn, const void *key, const void *value, const void *kv_cache,
                     const int32_t *slot_mapping, int num_tokens, int num_blocks, int block_size,
                     int num_kv_heads, int head_size, int dtype, long long *row_elems)
{
    if (dtype != PA_F16 && dtype != PA_BF16)
        return set_error(PA_ERR_UNSUPPORTED, "%s: dtype %d", fn, dtype);
    if (num_tokens < 0 || num_blocks <= 0 || block_size < kTile || block_size % kTile != 0 ||
        num_kv_heads <= 0 || head_size <= 0)
        return set_error(PA_ERR_INVALID_ARG, "%s: bad sizes", fn);
    if (((long long)num_kv_heads * head_size) % 8 != 0)
        return set_error(PA_ERR_INVALID_ARG, "%s: num_kv_heads * head_size must be a multiple of 8", fn);
    *row_elems = (long long)num_kv_heads * head_size;
    if (*row_elems > (1LL << 32))
        return set_error(PA_ERR_INVALID_ARG, "%s: row too large", fn);
    if (num_tokens == 0)
        return PA_OK;
    if (!key || !value || !kv_cache || !slot_mapping)
        return set_error(PA_ERR_INVALID_ARG, "%s: null pointer argument", fn);
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(kv_cache, 16) || !aligned(slot_mapping, 4))
        return set_error(PA_ERR_INVALID_ARG, "%s: misaligned pointer (16 B)", fn);
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_size, int block_size, int dtype, size_t *bytes)
{
    return workspace_size_impl("pa_decode_workspace_size", num_seqs, num_q_heads, num_kv_heads,
                               head_size, block_size, dtype, false, bytes);
}

extern "C" int pa_decode(void *out, const void *query, const void *kv_cache,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *seq_lens, int num_seqs, float scale, int num_q_heads,
                         int num_kv_heads, int head_size, int num_blocks, int block_size,
                         int dtype, void *workspace, size_t workspace_bytes, unsigned flags,
                         pa_stream_t stream)
{
    return decode_impl("pa_decode", out, query, kv_cache, block_tables, max_blocks_per_seq,
                       seq_lens, num_seqs, scale, num_q_heads, num_kv_heads, head_size, num_blocks,
                       block_size, dtype, false, 1.f, 1.f, workspace, workspace_bytes, flags, stream);
}

extern "C" int pa_decode_fp8_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                            int head_size, int block_size, int dtype,
                                            size_t *bytes)
{
    return workspace_size_impl("pa_decode_fp8_workspace_size", num_seqs, num_q_heads,
                               num_kv_heads, head_size, block_size, dtype, true, bytes);
}

extern "C" int pa_decode_fp8(void *out, const void *query, const void *kv_cache,
                             const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *seq_lens, int num_seqs, float scale, int num_q_heads,
                             int num_kv_heads, int head_size, int num_blocks, int block_size,
                             int dtype, float k_scale, float v_scale, void *workspace,
                             size_t workspace_bytes, unsigned flags, pa_stream_t stream)
{
    return decode_impl("pa_decode_fp8", out, query, kv_cache, block_tables, max_blocks_per_seq,
                       seq_lens, num_seqs, scale, num_q_heads, num_kv_heads, head_size, num_blocks,
                       block_size, dtype, true, k_scale, v_scale, workspace, workspace_bytes, flags,
                       stream);
}

extern "C" int pa_reshape_and_cache(const void *key, const void *value, void *kv_cache,
                                    const int32_t *slot_mapping, int num_tokens, int num_blocks,
                                    int block_size, int num_kv_heads, int head_size, int dtype,
                                    pa_stream_t stream)
{
    long long row_elems = 0;
    int rc = validate_reshape("pa_reshape_and_cache", key, value, kv_cache, slot_mapping, num_tokens,
                              num_blocks, block_size, num_kv_heads, head_size, dtype, &row_elems);
    if (rc != PA_OK || num_tokens == 0)
        return rc;
    const long long row_vecs = row_elems * 2 / 16;
    const long long num_slots = (long long)num_blocks * block_size;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Threads: a multiple of 32 covering the row in kReshapeVecs passes, at
    // most kReshapeMaxThreads (longer rows loop).
    const long long per = (row_vecs + kReshapeVecs - 1) / kReshapeVecs;
    const int threads = (int)std::min<long long>(kReshapeMaxThreads, (per + 31) / 32 * 32);
    reshape_and_cache_kernel<<<num_tokens, threads, 0, s>>>(
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
        static_cast<uint4 *>(kv_cache), slot_mapping, (int)row_vecs, num_slots, num_slots * row_vecs);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "pa_reshape_and_cache: launch");
    return PA_OK;
}

extern "C" int pa_reshape_and_cache_fp8(const void *key, const void *value, void *kv_cache,
                                        const int32_t *slot_mapping, int num_tokens,
                                        int num_blocks, int block_size, int num_kv_heads,
                                        int head_size, int dtype, float k_scale, float v_scale,
                                        pa_stream_t stream)
{
    long long row_elems = 0;
    int rc = validate_reshape("pa_reshape_and_cache_fp8", key, value, kv_cache, slot_mapping,
                              num_tokens, num_blocks, block_size, num_kv_heads, head_size, dtype,
                              &row_elems);
    if (rc != PA_OK)
        return rc;
    if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
        return set_error(PA_ERR_INVALID_ARG,
                         "pa_reshape_and_cache_fp8: k_scale and v_scale must be finite and > 0");
    if (num_tokens == 0)
        return PA_OK;
    const long long row_vecs = row_elems / 8;  // 8 elements: 16 bytes in, 8 bytes out
    const long long num_slots = (long long)num_blocks * block_size;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const dim3 grid(num_tokens, (unsigned)((row_vecs + kReshapeThreads - 1) / kReshapeThreads));
    if (dtype == PA_BF16)
        reshape_and_cache_fp8_kernel<true><<<grid, kReshapeThreads, 0, s>>>(
            static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
            static_cast<uint2 *>(kv_cache), slot_mapping, (int)row_vecs, num_slots,
            num_slots * row_vecs, k_scale, v_scale);
    else
        reshape_and_cache_fp8_kernel<false><<<grid, kReshapeThreads, 0, s>>>(
            static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
            static_cast<uint2 *>(kv_cache), slot_mapping, (int)row_vecs, num_slots,
            num_slots * row_vecs, k_scale, v_scale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "pa_reshape_and_cache_fp8: launch");
    return PA_OK;
}

extern "C" int pa_copy_blocks(void *const *kv_caches, int num_layers, const int32_t *src_dst_pairs,
                              int num_pairs, int num_blocks, int block_size, int num_kv_heads,
                              int head_size, int dtype, pa_stream_t stream)
{
    if (dtype != PA_F16 && dtype != PA_BF16 && dtype != PA_FP8_E4M3)
        return set_error(PA_ERR_UNSUPPORTED, "pa_copy_blocks: dtype %d", dtype);
    const long long esize = dtype == PA_FP8_E4M3 ? 1 : 2;
    if (num_pairs < 0 || num_layers < 1 || num_layers > kMaxLayers || num_blocks <= 0 ||
        block_size < kTile || block_size % kTile != 0 || num_kv_heads <= 0 || head_size <= 0)
        return set_error(PA_ERR_INVALID_ARG, "pa_copy_blocks: bad sizes (1 <= num_layers <= %d)", kMaxLayers);
    if (((long long)num_kv_heads * head_size * esize) % 16 != 0)
        return set_error(PA_ERR_INVALID_ARG, "pa_copy_blocks: a token's row (num_kv_heads * head_size elements) must be a multiple of 16 bytes");
    if (num_pairs == 0)
        return PA_OK;
    if (!kv_caches || !src_dst_pairs || !aligned(src_dst_pairs, 4))
        return set_error(PA_ERR_INVALID_ARG, "pa_copy_blocks: null or misaligned pointer argument");
    LayerPtrs lp;
    for (int l = 0; l < num_layers; ++l) {
        if (!kv_caches[l] || !aligned(kv_caches[l], 16))
            return set_error(PA_ERR_INVALID_ARG, "pa_copy_blocks: layer %d pool null or misaligned", l);
        lp.p[l] = static_cast<uint4 *>(kv_caches[l]);
    }
    for (int l = num_layers; l < kMaxLayers; ++l)
        lp.p[l] = nullptr;
    const long long block_vecs = (long long)block_size * num_kv_heads * head_size * esize / 16;
    const long long half_vecs = (long long)num_blocks * block_vecs;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    copy_blocks_kernel<<<dim3(num_pairs, num_layers), 256, 0, s>>>(lp, src_dst_pairs, num_pairs, num_blocks,
                                                                  block_vecs, half_vecs);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "pa_copy_blocks: launch");
    return PA_OK;
}

extern "C" int pa_get_device_error(int *bits)
{
    if (!bits)
        return set_error(PA_ERR_INVALID_ARG, "pa_get_device_error: bits is null");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cuda_fail(e, "pa_get_device_error: synchronize");
    int v = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int));
    if (e != cudaSuccess)
        return cuda_fail(e, "pa_get_device_error: read");
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    if (e != cudaSuccess)
        return cuda_fail(e, "pa_get_device_error: clear");
    int w = 0;
    e = static_cast<cudaError_t>(prefill_take_device_error(&w));
    if (e != cudaSuccess)
        return cuda_fail(e, "pa_get_device_error: prefill word");
    *bits = v | w;
    return PA_OK;
}
