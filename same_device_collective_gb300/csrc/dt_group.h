// The group object behind dt_group_t and the asynchronous work handle: host
// state of the same-device collective library.  Not part of the C ABI.
#pragma once

#include <atomic>
#include <condition_variable>
#include <cstdint>
#include <deque>
#include <mutex>
#include <vector>

#include "dt_internal.h"

struct dt_group;

// An asynchronous work: the end event of one async scope.
struct dt_work {
    dt_group *g = nullptr;
    cudaEvent_t end = nullptr;
};

// The group object behind dt_group_t.
struct dt_group {
    int P = 0;
    int device = 0;
    uint32_t timeout_ms = 2000;
    int64_t barriers_issued = 0;
    bool poisoned = false;
    dt_status poison_code = DT_OK;

    int32_t *d_win = nullptr;        // [P][P] window followed by rank_gen[P]
    dt::DevError *d_err = nullptr;
    dt::DevError *h_err = nullptr;   // host-mapped mirror (host view)
    dt::DevError *h_err_dev = nullptr;

    // bucket plans: pinned host buffers and device buffers.  A slot keeps the
    // arguments its plan was built for (key) and the launches it describes,
    // so a call with the same gradients, counts, dtype, op and cap reuses the
    // uploaded plan; a slot is rebuilt only after its event says the last
    // kernel reading it ended.  A slot used by a call under stream capture is
    // pinned: a CUDA graph holds its device address, so it is never rebuilt,
    // and new slots are added when every slot is pinned.
    struct PlanLaunch {
        size_t tb, te, start_off;
        uint64_t total, per_block;
        uint32_t blocks;
    };
    struct PlanSlot {
        void *h = nullptr;
        void *d = nullptr;
        size_t bytes = 0;
        cudaEvent_t done = nullptr;
        bool used = false;
        bool pinned = false;
        std::vector<uint64_t> key;
        std::vector<PlanLaunch> launches;
        size_t ptr_bytes = 0;
        size_t tab_bytes = 0;
    };
    static constexpr int kPlanSlots = 2;   // slots made at create
    std::deque<PlanSlot> plans;            // stable addresses as it grows
    int next_plan = 0;

    // rank-local calls: one host thread per rank meets the others here, like
    // the MemoryTensorStore of the DTorch page (mutex, condition variable,
    // CUDA events).  The last rank to arrive launches the group-wide kernel.
    struct RankCall {
        int kind;                 // which collective (dt_group.cpp: CallKind)
        const void *in;
        void *out;
        void *const *outv;        // AllGatherIntoVec: this rank's P outputs
        size_t count;             // elements / recv_count / this rank's rows / chunk bytes / R
        size_t row_bytes;         // row bytes / C (2-D AllToAll)
        int dtype, op;            // dtype or element bytes; op, shard index or src_dim
        int dim2;                 // dest_dim (2-D AllToAll)
        unsigned flags;
        cudaStream_t stream;
    };
    std::mutex rv_mu;
    std::condition_variable rv_cv;
    RankCall rv_call[DT_MAX_RANKS];
    bool rv_present[DT_MAX_RANKS] = {};
    int rv_arrived = 0;
    uint64_t rv_round = 0;
    bool rv_aborted = false;
    // bumped under rv_mu whenever rv_round or rv_aborted changes: waiting
    // ranks spin on it before they sleep on rv_cv
    std::atomic<uint64_t> rv_epoch{0};
    dt_status rv_status[2] = {DT_OK, DT_OK};
    cudaEvent_t rv_ready[DT_MAX_RANKS] = {};
    cudaEvent_t rv_done[2] = {nullptr, nullptr};
    cudaStream_t rv_launch[2] = {nullptr, nullptr};   // the stream round (parity) launched on

    // async scopes: the communication stream, the scope's start event and a
    // pool of work handles (each owns an end event)
    cudaStream_t comm = nullptr;
    cudaEvent_t scope_start = nullptr;
    bool scope_open = false;
    std::vector<dt_work *> work_free;
    std::vector<dt_work *> work_all;

    std::mutex mu;
};
