// rank_local_step: the rank-local ThreadGroup pattern driven from native threads.
//
// The ThreadGroup pages run one host thread per logical rank, each calling the
// collective for its own rank on its own stream ("DTorch ThreadGroup" §2, the
// MemoryTensorStore rendezvous of §3).  This program does exactly that through
// the C ABI's rank-local calls (rank >= 0): P std::threads, one CUDA stream
// each, run K steps of
//     barrier, ReduceScatter(avg), barrier, AllGather
// on one bf16 [rows, cols] input per rank, and it prints one JSON line with the
// wall time per step (both ends synchronised), the host time to issue a step,
// and the group's status.  No Python is involved, so the figure is the
// library's own rank-local cost.
//
// Usage: rank_local_step [P rows cols steps [shared]]   (defaults 4 8192 4096 2000)
//
// With "shared" every rank passes the same stream: the library then needs no
// cross-stream event waits at all, so the difference between the two runs is
// the cost of those waits.
//
// The inputs are filled with one constant: the step's memory traffic does not
// depend on the values, and the results are not checked here (the tests do).
#include <cuda_runtime.h>

#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <string>
#include <thread>
#include <vector>

#include "dt.h"

namespace {

int fail(const char *what, const char *detail)
{
    std::printf("{\"error\": \"%s: %s\"}\n", what, detail);
    return 1;
}

}  // namespace

int main(int argc, char **argv)
{
    const int P = argc > 1 ? std::atoi(argv[1]) : 4;
    const size_t rows = argc > 2 ? std::strtoull(argv[2], nullptr, 10) : 8192;
    const size_t cols = argc > 3 ? std::strtoull(argv[3], nullptr, 10) : 4096;
    const int steps = argc > 4 ? std::atoi(argv[4]) : 2000;
    const bool shared = argc > 5 && std::string(argv[5]) == "shared";
    if (P < 1 || P > DT_MAX_RANKS || rows == 0 || cols == 0 || rows % P || steps < 1)
        return fail("arguments", "need 1 <= P <= 16, rows % P == 0, steps >= 1");
    const size_t shard_rows = rows / P;
    const size_t in_bytes = rows * cols * 2, shard_bytes = shard_rows * cols * 2;

    dt_group_t g = nullptr;
    dt_status st = dt_group_create(P, 0, &g);
    if (st != DT_OK) return fail("dt_group_create", dt_status_string(st));

    std::vector<void *> xs(P, nullptr), rs(P, nullptr), ag(P, nullptr);
    std::vector<cudaStream_t> streams(P, nullptr);
    for (int r = 0; r < P; ++r) {
        cudaError_t e = cudaMalloc(&xs[r], in_bytes);
        if (e == cudaSuccess) e = cudaMalloc(&rs[r], shard_bytes);
        if (e == cudaSuccess) e = cudaMalloc(&ag[r], in_bytes);
        if (e == cudaSuccess) e = cudaMemset(xs[r], 0x3c, in_bytes);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&streams[r], cudaStreamNonBlocking);
        if (e != cudaSuccess) return fail("device setup", cudaGetErrorString(e));
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return fail("device setup", "synchronize");

    std::vector<int> bad(P, 0);
    auto run = [&](int k) {
        std::vector<std::thread> threads;
        for (int r = 0; r < P; ++r)
            threads.emplace_back([&, r] {
                if (cudaSetDevice(0) != cudaSuccess) { bad[r] = DT_ERR_CUDA; return; }
                void *s = streams[shared ? 0 : r];
                for (int i = 0; i < k && !bad[r]; ++i) {
                    int e = dt_barrier(g, r, s);
                    if (!e) e = dt_reduce_scatter(g, r, &xs[r], &rs[r], shard_rows * cols, DT_BF16,
                                                  DT_AVG, s);
                    if (!e) e = dt_barrier(g, r, s);
                    if (!e) e = dt_all_gather(g, r, &rs[r], &ag[r], nullptr, shard_rows, cols * 2, 0, s);
                    bad[r] = e;
                }
            });
        for (std::thread &t : threads) t.join();
    };

    run(20);   // warm-up
    if (cudaDeviceSynchronize() != cudaSuccess) return fail("warm-up", "synchronize");
    const auto t0 = std::chrono::steady_clock::now();
    run(steps);
    const auto t1 = std::chrono::steady_clock::now();
    const cudaError_t e = cudaDeviceSynchronize();
    const auto t2 = std::chrono::steady_clock::now();
    if (e != cudaSuccess) return fail("timed steps", cudaGetErrorString(e));
    for (int r = 0; r < P; ++r)
        if (bad[r]) return fail("rank call", dt_status_string((dt_status)bad[r]));
    const dt_status check = dt_group_check(g);

    const double wall_us = std::chrono::duration<double, std::micro>(t2 - t0).count() / steps;
    const double host_us = std::chrono::duration<double, std::micro>(t1 - t0).count() / steps;
    // ReduceScatter: P inputs read, P shards written; AllGather: P shards read, P outputs written
    const double bytes = (double)P * in_bytes + P * shard_bytes + P * shard_bytes + (double)P * in_bytes;
    std::printf("{\"P\": %d, \"rows\": %zu, \"cols\": %zu, \"steps\": %d, \"us_per_step\": %.2f, "
                "\"host_issue_us_per_step\": %.2f, \"GB/s\": %.1f, \"streams\": \"%s\", "
                "\"status_ok\": %s}\n",
                P, rows, cols, steps, wall_us, host_us, bytes / (wall_us * 1e-6) / 1e9,
                shared ? "one shared by all ranks" : "one per rank", check == DT_OK ? "true" : "false");

    for (int r = 0; r < P; ++r) {
        cudaStreamDestroy(streams[r]);
        cudaFree(xs[r]);
        cudaFree(rs[r]);
        cudaFree(ag[r]);
    }
    dt_group_destroy(g);
    return check == DT_OK ? 0 : 1;
}
