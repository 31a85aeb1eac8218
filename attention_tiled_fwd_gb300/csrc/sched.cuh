// sched.cuh -- work distribution of the persistent D = 64 forward
// (fwd_bf16_duo.cu).
//
// The TMA producer thread draws the CTA's work items and hands them to the
// CTA's other warps, in order, through a small ring in shared memory.  An item
// comes either from the static deal (persistent_work_index: round k of the
// work order dealt forwards and backwards in turn, which balances the CTAs
// when every round holds items of near-equal length) or from the launch's
// work counter (an atomic add per item: a CTA draws its next item as it
// issues the last loads of its current one, so the items go to the CTAs in
// the order they become free).  The counter is what lets the causal work
// order run by groups of heads: a group holds tiles of every length, and only
// first-come drawing balances such a sequence.
#pragma once
#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace fa {

constexpr int kWorkRing = 2;  // items in flight between the producer and the consumer warps (4, 8 no faster)

struct WorkRing {
    int *item;        // [kWorkRing] in shared memory
    uint64_t *full;   // [kWorkRing]: item k written (count 1, phase k / kWorkRing)
    uint64_t *empty;  // [kWorkRing]: every consumer warp has read item k (count = consumer warps)
};

// Producer: the k-th item of this CTA, -1 once the work is exhausted.
__device__ __forceinline__ int work_draw(const FwdArgs &a, int k, int n_work) {
    if (a.work == nullptr) return k * (int)gridDim.x < n_work ? persistent_work_index(k, n_work) : -1;
    const int L = atomicAdd(a.work, 1);
    return L < n_work ? L : -1;
}

// Producer: hand item k to the consumers once every consumer has read item k - kWorkRing from the same entry.
__device__ __forceinline__ bool work_publish(const WorkRing &r, int k, int L, int *status, int site) {
    const int s = k % kWorkRing;
    if (k >= kWorkRing && !mbar_wait(&r.empty[s], (k / kWorkRing - 1) & 1, status, site)) return false;
    r.item[s] = L;
    mbar_arrive(&r.full[s]);  // release: the item is visible to the warps that wait on this phase
    return true;
}

// Consumer warp (all 32 lanes): item k, or -1 with ok = false when the wait ran out.
__device__ __forceinline__ int work_take(const WorkRing &r, int k, int *status, int site, bool &ok) {
    const int s = k % kWorkRing;
    ok = warp_wait(&r.full[s], (k / kWorkRing) & 1, status, site);
    if (!ok) return -1;
    int L = 0;
    if ((threadIdx.x & 31) == 0) L = *reinterpret_cast<volatile int *>(&r.item[s]);
    L = __shfl_sync(0xffffffffu, L, 0);
    if ((threadIdx.x & 31) == 0) mbar_arrive(&r.empty[s]);
    return L;
}

// Producer, after its last draw (or an abandoned loop): the CTA has stopped drawing.  The last CTA to stop
// zeroes the counter for the next launch that is handed the same one; every CTA stops only after its last
// draw, so no draw of this launch can follow the reset.
__device__ __forceinline__ void work_finish(const FwdArgs &a) {
    if (a.work == nullptr) return;
    __threadfence();
    if (atomicAdd(a.work + 1, 1) == (int)gridDim.x - 1) {
        atomicExch(a.work, 0);
        atomicExch(a.work + 1, 0);
    }
}

}  // namespace fa
