// Host emulation, for the CPU tests, of what the library's CUDA-core kernels
// take from CUDA and from common.cuh. Compiled with SSA_HOST_EMULATION
// defined, a kernel file's kernels and C entry points build against this
// header with g++ (see tests/emu/*.cpp).
//
// Execution model. A launch runs its blocks one after another; the threads of
// a block are fibers (ucontext) on one host thread. A thread runs until it
// reaches a warp collective (a shuffle, vote, match or reduction, or
// __syncwarp) or __syncthreads, and there it waits. The scheduler resumes
// every runnable thread in turn. After each pass it completes every
// collective whose participants have all arrived: for a warp collective,
// every lane of its mask, waiting on a collective with the same mask; for
// __syncthreads, every thread of the block that has not exited. Completing a
// collective computes each participant's result, as the hardware would, and
// makes those threads runnable again. This follows CUDA's rules for code
// whose collectives name the lanes that reach them, divergent calls included
// (a vote by the whole warp, then a match among the lanes that voted yes). It
// also reports a deadlock, where the hardware would hang, as an error.
// Blocks run one at a time, so a function-local static array stands in for a
// block's shared memory, and atomics are plain operations.
#pragma once
#include <ucontext.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
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

struct uint2 { uint32_t x, y; };
struct uint4 { uint32_t x, y, z, w; };
struct int4 { int32_t x, y, z, w; };
struct float4 { float x, y, z, w; };
inline float4 make_float4(float a, float b, float c, float d) { return {a, b, c, d}; }
inline uint4 make_uint4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) { return {a, b, c, d}; }
inline int4 make_int4(int32_t a, int32_t b, int32_t c, int32_t d) { return {a, b, c, d}; }

struct emu_dim { unsigned x = 0; };

namespace emu {

enum Op { NONE = 0, SHFL, BALLOT, MATCH_ANY, RED_OR, RED_AND, RED_ADD, SYNCWARP, SYNCTHREADS };

struct Thread {
    ucontext_t ctx;
    bool done = false;
    Op op = NONE;           // the collective it waits on (NONE: runnable)
    unsigned mask = 0;      // its lanes (warp collectives)
    uint64_t val = 0;       // its contribution
    int src = 0;            // shuffles: the source lane
    uint64_t res = 0;       // the result, once completed
};

struct Block {
    ucontext_t sched;
    std::vector<Thread> th;
    std::vector<char> stacks;
    unsigned n = 0, cur = 0;
    void (*entry)(void*) = nullptr;
    void* arg = nullptr;
};

inline Block* blk = nullptr;
inline emu_dim tid, bid, bdim, gdim;
constexpr size_t kStack = 128 << 10;

inline unsigned lane() { return tid.x & 31u; }

inline void thread_main() {
    blk->entry(blk->arg);
    blk->th[blk->cur].done = true;   // returning switches to uc_link (the scheduler)
}

// Waits on a collective; returns this thread's result.
inline uint64_t wait(Op op, unsigned mask, uint64_t val, int src = 0) {
    Thread& t = blk->th[blk->cur];
    t.op = op;
    t.mask = mask;
    t.val = val;
    t.src = src;
    swapcontext(&t.ctx, &blk->sched);
    return blk->th[blk->cur].res;
}

// Completes the collectives of warp w whose participants have all arrived.
inline bool complete_warp(unsigned w) {
    bool any = false;
    Thread* T = blk->th.data() + 32 * w;
    const unsigned nl = std::min(32u, blk->n - 32 * w);
    for (unsigned l = 0; l < nl; ++l) {
        const Op op = T[l].op;
        if (op == NONE || op == SYNCTHREADS || T[l].done) continue;
        const unsigned m = T[l].mask;
        bool ready = true;
        for (unsigned q = 0; q < nl && ready; ++q)
            if ((m >> q) & 1u) ready = !T[q].done && T[q].op == op && T[q].mask == m;
        if (!ready) continue;
        uint64_t ballot = 0, red_or = 0, red_and = ~0ull, red_add = 0;
        for (unsigned q = 0; q < nl; ++q) {
            if (!((m >> q) & 1u)) continue;
            if (T[q].val) ballot |= 1ull << q;
            red_or |= T[q].val;
            red_and &= T[q].val;
            red_add += T[q].val;
        }
        for (unsigned q = 0; q < nl; ++q) {
            if (!((m >> q) & 1u)) continue;
            Thread& P = T[q];
            switch (op) {
                case SHFL: {
                    const unsigned s = (unsigned)P.src & 31u;
                    P.res = ((m >> s) & 1u) ? T[s].val : P.val;   // a lane outside the mask: own value
                    break;
                }
                case BALLOT: P.res = ballot; break;
                case MATCH_ANY: {
                    uint64_t mm = 0;
                    for (unsigned r = 0; r < nl; ++r)
                        if (((m >> r) & 1u) && T[r].val == P.val) mm |= 1ull << r;
                    P.res = mm;
                    break;
                }
                case RED_OR: P.res = red_or; break;
                case RED_AND: P.res = red_and; break;
                case RED_ADD: P.res = red_add; break;
                default: P.res = 0; break;
            }
        }
        for (unsigned q = 0; q < nl; ++q)
            if ((m >> q) & 1u) T[q].op = NONE;
        any = true;
    }
    return any;
}

// Runs body() for every thread of every block; aborts on a deadlock.
template <typename F>
void launch(unsigned grid, unsigned block, F& body) {
    gdim.x = grid;
    bdim.x = block;
    Block B;
    B.n = block;
    B.th.resize(block);
    B.stacks.resize(kStack * block);
    B.entry = [](void* a) { (*static_cast<F*>(a))(); };
    B.arg = &body;
    blk = &B;
    for (unsigned b = 0; b < grid; ++b) {
        bid.x = b;
        for (unsigned t = 0; t < block; ++t) {
            Thread& T = B.th[t];
            T = Thread();
            getcontext(&T.ctx);
            T.ctx.uc_stack.ss_sp = B.stacks.data() + kStack * t;
            T.ctx.uc_stack.ss_size = kStack;
            T.ctx.uc_link = &B.sched;
            makecontext(&T.ctx, thread_main, 0);
        }
        for (;;) {
            bool ran = false, live = false;
            for (unsigned t = 0; t < block; ++t) {
                Thread& T = B.th[t];
                if (T.done) continue;
                live = true;
                if (T.op != NONE) continue;
                B.cur = t;
                tid.x = t;
                swapcontext(&B.sched, &T.ctx);
                ran = true;
            }
            if (!live) break;
            bool progressed = false;
            for (unsigned w = 0; w * 32 < block; ++w) progressed |= complete_warp(w);
            // __syncthreads: every thread that has not exited is waiting on it
            bool all_sync = true, some_sync = false;
            for (unsigned t = 0; t < block; ++t) {
                if (B.th[t].done) continue;
                if (B.th[t].op == SYNCTHREADS)
                    some_sync = true;
                else
                    all_sync = false;
            }
            if (all_sync && some_sync) {
                for (unsigned t = 0; t < block; ++t)
                    if (!B.th[t].done) B.th[t].op = NONE;
                progressed = true;
            }
            if (!ran && !progressed) {
                std::fprintf(stderr, "emulation: deadlock in block %u\n", b);
                std::abort();
            }
        }
    }
    blk = nullptr;
}

template <typename T>
inline uint64_t bits(T v) {
    static_assert(sizeof(T) <= 8, "at most 8 bytes");
    uint64_t b = 0;
    std::memcpy(&b, &v, sizeof(T));
    return b;
}
template <typename T>
inline T from_bits(uint64_t b) {
    T v;
    std::memcpy(&v, &b, sizeof(T));
    return v;
}

}  // namespace emu

// tid is set by the scheduler before each resume, so it is the running thread's
#define threadIdx (emu::tid)
#define blockIdx (emu::bid)
#define blockDim (emu::bdim)
#define gridDim (emu::gdim)

template <typename T>
inline T __shfl_sync(unsigned m, T v, int src) {
    return emu::from_bits<T>(emu::wait(emu::SHFL, m, emu::bits(v), src));
}
template <typename T>
inline T __shfl_xor_sync(unsigned m, T v, int o) {
    return __shfl_sync(m, v, (int)(emu::lane() ^ (unsigned)o));
}
template <typename T>
inline T __shfl_up_sync(unsigned m, T v, unsigned d) {
    const int s = (int)emu::lane() - (int)d;
    return __shfl_sync(m, v, s < 0 ? (int)emu::lane() : s);
}
template <typename T>
inline T __shfl_down_sync(unsigned m, T v, unsigned d) {
    const int s = (int)emu::lane() + (int)d;
    return __shfl_sync(m, v, s > 31 ? (int)emu::lane() : s);
}
inline unsigned __ballot_sync(unsigned m, int p) {
    return (unsigned)emu::wait(emu::BALLOT, m, p ? 1u : 0u);
}
inline int __any_sync(unsigned m, int p) { return __ballot_sync(m, p) != 0; }
inline int __all_sync(unsigned m, int p) { return __ballot_sync(m, p) == (m & 0xffffffffu); }
template <typename T>
inline unsigned __match_any_sync(unsigned m, T v) {
    return (unsigned)emu::wait(emu::MATCH_ANY, m, emu::bits(v));
}
inline unsigned __reduce_or_sync(unsigned m, unsigned v) {
    return (unsigned)emu::wait(emu::RED_OR, m, v);
}
inline unsigned __reduce_and_sync(unsigned m, unsigned v) {
    return (unsigned)emu::wait(emu::RED_AND, m, v);
}
inline unsigned __reduce_add_sync(unsigned m, unsigned v) {
    return (unsigned)emu::wait(emu::RED_ADD, m, v);
}
inline void __syncwarp(unsigned m = 0xffffffffu) { emu::wait(emu::SYNCWARP, m, 0); }
inline void __syncthreads() { emu::wait(emu::SYNCTHREADS, 0, 0); }
inline int __popc(unsigned v) { return __builtin_popcount(v); }
inline int __popcll(unsigned long long v) { return __builtin_popcountll(v); }
inline int __ffs(unsigned v) { return __builtin_ffs((int)v); }
inline int __clz(unsigned v) { return v ? __builtin_clz(v) : 32; }
template <typename T>
inline T __ldg(const T* p) { return *p; }
inline int atomicAdd(int* p, int v) { int o = *p; *p = o + v; return o; }
inline unsigned atomicAdd(unsigned* p, unsigned v) { unsigned o = *p; *p = o + v; return o; }
inline int atomicOr(int* p, int v) { int o = *p; *p = o | v; return o; }
inline unsigned atomicMax(unsigned* p, unsigned v) { unsigned o = *p; *p = std::max(o, v); return o; }
inline float __uint_as_float(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }
inline uint32_t __float_as_uint(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }
inline float __fsub_rn(float a, float b) { return a - b; }
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

inline uint4 ld_nc_na16(const void* p) { return ldg16(p); }

// order keys, head map and selection keys, as in the library's common.cuh
inline uint32_t f32_order_key(float f) {
    uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
inline float order_key_f32(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}
struct HeadMap {
    int H, H_kv, H_idx;
    int grouped, head_inner;
};
inline uint64_t sel_key(uint32_t okey, uint32_t j) {
    return (static_cast<uint64_t>(okey) << 32) | static_cast<uint64_t>(~j);
}
inline uint32_t sel_key_index(uint64_t key) { return ~static_cast<uint32_t>(key); }
inline uint32_t sel_key_okey(uint64_t key) { return static_cast<uint32_t>(key >> 32); }

struct TraceLaunch {   // launch tracing is a no-op here
    TraceLaunch(const char*, cudaStream_t) {}
};
}  // namespace ssa

// bf16 storage: the high half of an fp32, rounded to nearest even (finite
// inputs; NaN stays a NaN)
struct __nv_bfloat16 {
    uint16_t x;
};
struct __nv_bfloat162 {
    __nv_bfloat16 x, y;
};
inline __nv_bfloat16 emu_f32_to_bf16(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return {(uint16_t)((u >> 16) | 0x40u)};
    u += 0x7FFFu + ((u >> 16) & 1u);
    return {(uint16_t)(u >> 16)};
}
inline __nv_bfloat162 __floats2bfloat162_rn(float a, float b) {
    return {emu_f32_to_bf16(a), emu_f32_to_bf16(b)};
}
