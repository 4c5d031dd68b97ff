// Throughput and issue behaviour of single-SM tcgen05 MMAs (kind::f16, bf16,
// M = 128, K = 16, both operands in shared memory), one CTA per SM on every
// SM, the accumulator in tensor memory.
//
//   part 1: one issuing thread, N = 64, 128, 256: cycles per MMA and
//           FLOP/cycle/SM (the chunked-prefill MMAs are N = 128);
//   part 2: N = 128 with 1, 2 or 4 issuing warps, each issuing groups of 8
//           MMAs with a spin of G cycles between groups (the work an issuing
//           thread does between its MMA groups): cycles per MMA overall,
//           and when the first group's issues returned.
//
// Build and run: nvcc -O3 -gencode arch=compute_103a,code=sm_103a tcgen05_issue.cu -o tcgen05_issue && ./tcgen05_issue
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <vector>

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t gtimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t ph)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.b32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(ph)
                 : "memory");
    return ok;
}

// Bounded: gives up after one second (the caller records an error).
__device__ bool mbar_wait(uint32_t bar, uint32_t ph)
{
    const uint64_t t0 = gtimer();
    while (!mbar_try(bar, ph))
        if (gtimer() - t0 > 1000000000ull)
            return false;
    return true;
}

// Shared-memory matrix descriptor: start, leading and stride byte offsets
// (16-byte units), version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__device__ __forceinline__ uint32_t idesc(int m, int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, 1, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                 "l"(a), "l"(b), "r"(id)
                 : "memory");
}

__device__ __forceinline__ void commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void spin(long long c)
{
    const long long t = clock64();
    while (clock64() - t < c) {
    }
}

constexpr int kOperandBytes = 32768 + 65536;  // A: 128 x 128 bf16; B: up to 256 x 128 bf16

// nwarps issuing warps (lane 0 each) issue `groups` groups of 8 MMAs of
// 128 x n x 16 into their own accumulator, spinning `gap` cycles between
// groups. cyc[cta] = cycles from the start until every MMA has completed.
__global__ void __launch_bounds__(128) issue(long long *cyc, long long *ts, int *err, int n, int nwarps, int gap,
                                             int groups)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    __shared__ uint64_t bar[4];
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t *sm = smem_raw + (base - raw);
    for (int i = tid * 16; i < kOperandBytes; i += 128 * 16)
        *reinterpret_cast<uint4 *>(sm + i) = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int i = 0; i < 4; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[i])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tmem_base))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const long long t0 = clock64();
    if (lane == 0 && warp < nwarps) {
        const uint32_t id = idesc(128, n), sA = base, sB = base + 32768, bchunk = (uint32_t)n * 128;
        const uint32_t d = tmem_base + (uint32_t)(128 * warp);  // 4 x 128 columns at most (n <= 128 then)
        for (int g = 0; g < groups; ++g) {
            for (int k = 0; k < 8; ++k) {
                mma(d, desc(sA + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
                    desc(sB + (k >> 2) * bchunk + (k & 3) * 32, 16, 1024), id);
                if (g == 0 && blockIdx.x == 0)
                    ts[warp * 8 + k] = clock64() - t0;
            }
            if (gap > 0)
                spin(gap);
        }
        commit(smem_u32(&bar[warp]));
        if (!mbar_wait(smem_u32(&bar[warp]), 0))
            atomicOr(err, 1);
    }
    __syncthreads();
    if (tid == 0)
        cyc[blockIdx.x] = clock64() - t0;
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base) : "memory");
}

int main()
{
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    long long *dc, *dts;
    int *derr;
    if (cudaMalloc(&dc, sizeof(long long) * 1024) != cudaSuccess || cudaMalloc(&dts, sizeof(long long) * 64) ||
        cudaMalloc(&derr, 4))
        return 1;
    const int smem = kOperandBytes + 1024 + 60000;  // more than half an SM's shared memory: one CTA per SM
    cudaFuncSetAttribute(issue, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    auto run = [&](int n, int nw, int gap, int groups) {
        cudaMemset(derr, 0, 4);
        for (int rep = 0; rep < 2; ++rep)
            issue<<<sms, 128, smem>>>(dc, dts, derr, n, nw, gap, groups);
        if (cudaDeviceSynchronize() != cudaSuccess)
            return false;
        std::vector<long long> c(sms), t(64);
        int herr = 0;
        cudaMemcpy(c.data(), dc, sizeof(long long) * sms, cudaMemcpyDeviceToHost);
        cudaMemcpy(t.data(), dts, sizeof(long long) * 64, cudaMemcpyDeviceToHost);
        cudaMemcpy(&herr, derr, 4, cudaMemcpyDeviceToHost);
        double mean = 0;
        for (auto v : c)
            mean += v;
        mean /= sms;
        const double per = mean / (groups * 8.0 * nw);
        printf("{\"N\": %d, \"issuing_warps\": %d, \"gap_cycles\": %d, \"err\": %d, \"cycles_per_mma\": %.1f, "
               "\"flop_per_cycle_per_sm\": %.0f, \"first_group_issue_cycles\": [",
               n, nw, gap, herr, per, 2.0 * 128 * n * 16 / per);
        for (int k = 0; k < 8; ++k)
            printf("%s%lld", k ? ", " : "", t[k]);
        printf("]}\n");
        return true;
    };
    for (int n : {64, 128, 256})
        if (!run(n, 1, 0, 512))
            return 1;
    for (int nw : {1, 2, 4})
        for (int gap : {0, 300, 1000})
            if (!run(128, nw, gap, 256))
                return 1;
    return 0;
}
