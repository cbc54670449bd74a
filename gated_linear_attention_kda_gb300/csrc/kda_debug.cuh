// kda_debug.cuh -- the device error word shared by every kernel of the library, and the bounds
// checks of the debug build.
//
// With KDA_DEBUG defined (libkda_debug.so) every shared-memory, tensor-memory, TMA and global
// access of the forward kernels is checked before it is made: an access outside its buffer sets
// DEVERR_BOUNDS in the device error word (reported by kda_check_device_status) and is skipped,
// so a wrong index shows up as an error status instead of a fault. Warp-collective accesses
// (ldmatrix, stmatrix) are skipped by the whole warp when any lane is out of bounds; tensor-memory
// accesses are only flagged (their addresses are warp-uniform). Without KDA_DEBUG every check is
// the constant `true` and compiles away.
#pragma once
#include <cstdint>

namespace kda {

enum : unsigned { DEVERR_SEQLENS = 1u, DEVERR_TIMEOUT = 2u, DEVERR_BOUNDS = 4u };
__device__ unsigned int g_dev_error;

#ifdef KDA_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// The start of the dynamic shared memory window: dynamic shared memory follows the static one,
// so [0, this + %dynamic_smem_size) bounds every shared address of the CTA.
extern __shared__ uint8_t kda_dynamic_smem[];

__device__ __forceinline__ uint32_t dbg_smem_end()
{
    uint32_t n;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(n));
    return static_cast<uint32_t>(__cvta_generic_to_shared(kda_dynamic_smem)) + n;
}

__device__ __forceinline__ bool dbg_flag(bool ok)
{
    if (!ok) atomicOr(&g_dev_error, DEVERR_BOUNDS);
    return ok;
}

// `bytes` at shared address `addr` lie inside the CTA's shared memory
__device__ __forceinline__ bool smem_ok(uint32_t addr, uint32_t bytes)
{
    if constexpr (!kDebugChecks) return true;
    const uint64_t end = static_cast<uint64_t>(addr) + bytes;
    return dbg_flag(end <= dbg_smem_end());
}

// the same for a warp-collective access: true when every lane's access is inside
__device__ __forceinline__ bool smem_ok_warp(uint32_t addr, uint32_t bytes)
{
    if constexpr (!kDebugChecks) return true;
    return __all_sync(0xffffffffu, smem_ok(addr, bytes));
}

// a shared address used through the kernels' SM_AT accessor: itself when inside, else `safe`
// (the CTA's shared base) after flagging
__device__ __forceinline__ uint32_t smem_checked(uint32_t addr, uint32_t bytes, uint32_t safe)
{
    if constexpr (!kDebugChecks) return addr;
    return smem_ok(addr, bytes) ? addr : safe;
}

// `n` consecutive tensor-memory columns from address `taddr` (lane << 16 | column) lie inside the
// 512 columns of an SM; flagged only
__device__ __forceinline__ void tmem_check(uint32_t taddr, uint32_t n)
{
    if constexpr (kDebugChecks) dbg_flag((taddr & 0xffffu) + n <= 512u && (taddr >> 16) < 128u);
}

// elements [idx, idx + n) of a global buffer of `limit` elements
__device__ __forceinline__ bool gmem_ok(size_t idx, size_t n, size_t limit)
{
    if constexpr (!kDebugChecks) return true;
    return dbg_flag(idx + n <= limit);
}

}  // namespace kda
