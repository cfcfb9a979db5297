// Host emulation, for the CPU tests, of what the backward kernels
// (dynamic_top_sparse_rank_b300/csrc/attn_bwd.cu) take from CUDA and from the
// library's common.cuh. Compiled with SSA_HOST_EMULATION defined, the kernels
// and the C entry points of attn_bwd.cu build against this header with g++.
//
// Execution model. A launch runs its blocks one after another. The threads of
// a block are fibers (ucontext) on one host thread. A barrier (__syncwarp,
// __syncthreads, and each of the two halves of a shuffle) switches back to
// the scheduler. The scheduler resumes every live thread in turn, so each
// pass advances every thread to its next barrier. This is exact for code in
// which the threads of a warp (or of the block, for __syncthreads) meet the
// same barriers in the same order, as warp-synchronous CUDA code must. It
// also holds when a whole warp returns early: its threads just stop taking
// part. A shuffle stores the value in the warp's slot table before its first
// barrier and reads the source lane's slot after it. Blocks run one at a
// time, so a function-local static array stands in for a block's shared
// memory. The bf16 and vector helpers restate the library's (bf16 is the high
// half of an fp32). Runtime calls act on host memory.
#pragma once
#include <ucontext.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <math.h>
#include <vector>

#include "ssa.h"

#define __global__
#define __device__
#define __host__
#define __forceinline__ inline
#define __launch_bounds__(...)
#define __shared__ static
#define SSA_DEVINL inline

struct uint4 { uint32_t x, y, z, w; };
struct float4 { float x, y, z, w; };
inline float4 make_float4(float a, float b, float c, float d) { return {a, b, c, d}; }
inline uint4 make_uint4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) { return {a, b, c, d}; }

struct emu_dim { unsigned x = 0; };

namespace emu {

struct Thread {
    ucontext_t ctx;
    bool done = false;
};

struct Block {
    ucontext_t sched;
    std::vector<Thread> th;
    std::vector<char> stacks;
    std::vector<uint64_t> slot;   // one 32-entry table per warp
    unsigned cur = 0;
    void (*entry)(void*) = nullptr;
    void* arg = nullptr;
};

inline Block* blk = nullptr;
inline emu_dim tid, bid, bdim, gdim;
constexpr size_t kStack = 256 << 10;

inline void yield() {
    Thread& t = blk->th[blk->cur];
    swapcontext(&t.ctx, &blk->sched);
}

inline void thread_main() {
    blk->entry(blk->arg);
    blk->th[blk->cur].done = true;
    // returning switches to uc_link (the scheduler)
}

// Runs body() for every thread of every block.
template <typename F>
void launch(unsigned grid, unsigned block, F& body) {
    gdim.x = grid;
    bdim.x = block;
    Block B;
    B.th.resize(block);
    B.stacks.resize(kStack * block);
    B.slot.assign(((block + 31) / 32) * 32, 0);
    B.entry = [](void* a) { (*static_cast<F*>(a))(); };
    B.arg = &body;
    blk = &B;
    for (unsigned b = 0; b < grid; ++b) {
        bid.x = b;
        for (unsigned t = 0; t < block; ++t) {
            Thread& T = B.th[t];
            T.done = false;
            getcontext(&T.ctx);
            T.ctx.uc_stack.ss_sp = B.stacks.data() + kStack * t;
            T.ctx.uc_stack.ss_size = kStack;
            T.ctx.uc_link = &B.sched;
            makecontext(&T.ctx, thread_main, 0);
        }
        for (bool live = true; live;) {
            live = false;
            for (unsigned t = 0; t < block; ++t) {
                if (B.th[t].done) continue;
                B.cur = t;
                tid.x = t;
                swapcontext(&B.sched, &B.th[t].ctx);
                live |= !B.th[t].done;
            }
        }
    }
    blk = nullptr;
}

inline unsigned lane() { return tid.x & 31u; }
inline uint64_t* warp_slots() { return blk->slot.data() + (tid.x & ~31u); }

}  // namespace emu

// tid is set by the scheduler before each resume, so it is the running thread's
#define threadIdx (emu::tid)
#define blockIdx (emu::bid)
#define blockDim (emu::bdim)
#define gridDim (emu::gdim)

template <typename T>
inline T __shfl_sync(unsigned, T v, int src) {
    static_assert(sizeof(T) <= 8, "shuffle of at most 8 bytes");
    uint64_t b = 0;
    std::memcpy(&b, &v, sizeof(T));
    uint64_t* slots = emu::warp_slots();
    slots[emu::lane()] = b;
    emu::yield();
    const uint64_t r = emu::warp_slots()[src & 31];
    emu::yield();
    T out;
    std::memcpy(&out, &r, sizeof(T));
    return out;
}
template <typename T>
inline T __shfl_xor_sync(unsigned m, T v, int o) {
    return __shfl_sync(m, v, (int)(emu::lane() ^ (unsigned)o));
}
inline void __syncwarp(unsigned = 0xffffffffu) { emu::yield(); }
inline void __syncthreads() { emu::yield(); }
template <typename T>
inline T __ldg(const T* p) { return *p; }
inline int atomicAdd(int* p, int v) { int o = *p; *p = o + v; return o; }   // one host thread
inline int atomicOr(int* p, int v) { int o = *p; *p = o | v; return o; }
inline float __uint_as_float(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }
using std::max;
using std::min;

// the runtime calls the launch code makes, on host memory
typedef int cudaError_t;
typedef void* cudaStream_t;
enum { cudaSuccess = 0, cudaErrorInvalidValue = 1, cudaErrorInvalidConfiguration = 9 };
inline cudaError_t cudaMemsetAsync(void* p, int v, size_t n, cudaStream_t) {
    std::memset(p, v, n);
    return cudaSuccess;
}
inline cudaError_t cudaGetLastError() { return cudaSuccess; }

template <typename F>
void emu_launch(unsigned grid, unsigned block, F&& body) {
    emu::launch(grid, block, body);
}

namespace ssa {
constexpr float kLog2e = 1.4426950408889634f;
inline void report(int32_t* dev_status, int bit) {
    if (dev_status) atomicOr(dev_status, bit);
}
inline void bf16x8_to_f32(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
inline void f32x4_to_f32(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}
template <bool BF16>
struct Vec16 {
    static constexpr int E = BF16 ? 8 : 4;
    static void to_f32(const uint4& v, float* f) {
        if constexpr (BF16)
            bf16x8_to_f32(v, f);
        else
            f32x4_to_f32(v, f);
    }
};
inline uint4 ldg16(const void* p) {
    uint4 r;
    std::memcpy(&r, p, 16);
    return r;
}

struct TraceLaunch {   // launch tracing is a no-op here
    TraceLaunch(const char*, cudaStream_t) {}
};
}  // namespace ssa
