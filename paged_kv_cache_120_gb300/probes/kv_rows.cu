// Bandwidth ceiling of the paged K/V access pattern, by row size.
//
// A decode tile reads, for one kv head, 16 token rows of R bytes from K and
// the same from V; consecutive token rows of a head are H * R bytes apart
// (H kv heads per token row of the pool, R = head_size x element size), and
// each tile's block is a random one of the pool. This program reads ~1.2 GB
// per launch in exactly that pattern with plain 16-byte loads (no shared
// memory, no compute) and reports GB/s for R = 64..512 at H = 40 and H = 8:
// the most a kernel that reads those rows can expect from HBM. A 16-bit
// cache at head size 128 has R = 256; an FP8 cache has R = 128.
//
// Build and run: nvcc -O3 -gencode arch=compute_103a,code=sm_103a kv_rows.cu -o kv_rows && ./kv_rows
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <random>
#include <vector>

__global__ void read_rows(const uint4 *__restrict__ pool, const int *__restrict__ blk, long long ntiles,
                          int H, int R, long long S, long long half, unsigned *sink)
{
    const int lane = threadIdx.x & 31;
    const long long gw = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const long long nw = (gridDim.x * (long long)blockDim.x) >> 5;
    const int vec_per_row = R / 16;
    const int vec_per_tile = 2 * 16 * vec_per_row;  // K rows, then V rows
    unsigned acc = 0;
    for (long long t = gw; t < ntiles; t += nw) {
        const long long b = blk[t];
        const int h = (int)(t % H);
        for (int v = lane; v < vec_per_tile; v += 32) {
            const int c = v / (16 * vec_per_row);
            const int rem = v - c * 16 * vec_per_row;
            const int row = rem / vec_per_row, col = rem - row * vec_per_row;
            const long long byte = c * half + b * 16 * S + row * S + (long long)h * R + col * 16;
            const uint4 x = __ldcs(pool + byte / 16);
            acc ^= x.x ^ x.y ^ x.z ^ x.w;
        }
    }
    if (acc == 0x12345678u)
        sink[0] = acc;  // keeps the loads alive
}

int main()
{
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    const long long total = 3LL << 30;  // a 3 GiB pool: far larger than L2
    uint4 *pool = nullptr;
    unsigned *sink = nullptr;
    if (cudaMalloc(&pool, total) != cudaSuccess || cudaMalloc(&sink, 4) != cudaSuccess) {
        printf("{\"error\": \"allocation failed\"}\n");
        return 1;
    }
    cudaMemset(pool, 1, total);
    for (int H : {40, 8}) {
        for (int R : {64, 128, 256, 512}) {
            const long long S = (long long)H * R;
            const long long half = total / 2 / (16 * S) * (16 * S);  // K half, then V half
            const long long NB = half / (16 * S);
            const long long ntiles = (1200LL << 20) / (2 * 16 * R);
            // the largest byte any thread reads must lie inside the pool
            const long long last = half + (NB - 1) * 16 * S + 15 * S + (long long)(H - 1) * R + R;
            if (last > total) {
                printf("{\"error\": \"bounds\"}\n");
                return 1;
            }
            std::vector<int> blk(ntiles);
            std::mt19937_64 g(1);
            for (auto &x : blk)
                x = (int)(g() % NB);
            int *dblk = nullptr;
            if (cudaMalloc(&dblk, ntiles * sizeof(int)) != cudaSuccess)
                return 1;
            cudaMemcpy(dblk, blk.data(), ntiles * sizeof(int), cudaMemcpyHostToDevice);
            const int threads = 384, grid = sms * 4;
            cudaEvent_t a, b;
            cudaEventCreate(&a);
            cudaEventCreate(&b);
            for (int i = 0; i < 3; ++i)
                read_rows<<<grid, threads>>>(pool, dblk, ntiles, H, R, S, half, sink);
            const int reps = 10;
            cudaEventRecord(a);
            for (int i = 0; i < reps; ++i)
                read_rows<<<grid, threads>>>(pool, dblk, ntiles, H, R, S, half, sink);
            cudaEventRecord(b);
            cudaEventSynchronize(b);
            float ms = 0;
            cudaEventElapsedTime(&ms, a, b);
            const double bytes = (double)ntiles * 2 * 16 * R;
            printf("{\"H\": %d, \"R\": %d, \"bytes_per_launch\": %.0f, \"us_per_launch\": %.1f, "
                   "\"GBps\": %.0f, \"err\": \"%s\"}\n",
                   H, R, bytes, 1e3 * ms / reps, bytes * reps / (ms / 1e3) / 1e9,
                   cudaGetErrorString(cudaGetLastError()));
            cudaEventDestroy(a);
            cudaEventDestroy(b);
            cudaFree(dblk);
        }
    }
    cudaFree(pool);
    cudaFree(sink);
    return 0;
}
