// common.cuh -- device helpers shared by the library's kernels (sm_103a).
//
// Inline PTX for: mbarrier pipelines with bounded waits, 1-D bulk and 4-D tiled
// TMA copies into shared memory, programmatic dependent launch, warp-level
// tensor-core MMA (m16n8k16, fp32 accumulate) and ldmatrix.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gattn {

// Device status word bits (read and cleared by gattn_layer_poll_status).
enum : unsigned { kStatusRange = 1u, kStatusTimeout = 2u };

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Kernel arguments live in a constant bank that each SM caches; the first read
// of an argument misses and waits for a fill from L2, about a microsecond under
// load.  arg_fold() combines argument values into one word; a kernel stores it
// to a scratch word of shared memory before its grid dependency wait, so that
// the fills happen during the wait and the reads after it hit the cache.
__device__ __forceinline__ unsigned arg_bits(int v) { return (unsigned)v; }
__device__ __forceinline__ unsigned arg_bits(unsigned v) { return v; }
__device__ __forceinline__ unsigned arg_bits(float v) { return __float_as_uint(v); }
__device__ __forceinline__ unsigned arg_bits(long long v) { return (unsigned)v ^ (unsigned)(v >> 32); }
__device__ __forceinline__ unsigned arg_bits(unsigned long long v)
{
    return (unsigned)v ^ (unsigned)(v >> 32);
}
__device__ __forceinline__ unsigned arg_bits(const void *p)
{
    return arg_bits((unsigned long long)p);
}
template <class... T>
__device__ __forceinline__ unsigned arg_fold(const T &...v)
{
    return (arg_bits(v) ^ ... ^ 0u);
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity.  Gives up after limit_ns, or at
// once when *abort is already set; on giving up it sets *abort and the status
// word's timeout bit and returns false.  Callers keep their control flow (every
// named barrier is still reached) and skip the work of an aborted stage.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          unsigned *status,
                                          unsigned long long limit_ns = kWaitLimitNs)
{
    if (mbar_try(bar, parity))
        return true;
    if (*abort)
        return false;
    unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_try(bar, parity))
            return true;
        if (*abort)
            return false;
        if (global_ns() - t0 > limit_ns) {
            *abort = 1;
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

// Wait for the phase with the given parity, bounded by `limit_ns` but not cut
// short by an abort flag: for barriers whose completion must be observed
// before the thread goes on (bytes other CTAs are still sending here).  Sets
// the status word's timeout bit and returns false if the limit passes.
__device__ __forceinline__ bool mbar_wait_all(uint64_t *bar, uint32_t parity, unsigned *status,
                                              unsigned long long limit_ns)
{
    if (mbar_try(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try(bar, parity)) {
        if (global_ns() - t0 > limit_ns) {
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------- TMA copies

__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                        uint64_t policy)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
                 : "memory");
}

// Copies N (4, 8 or 16) bytes global -> shared without making the issuing
// thread wait (cp.async); cp_async_wait_all() waits for every copy the thread
// issued before it.  Both addresses aligned to N.
template <int N>
__device__ __forceinline__ void cp_async(void *dst, const void *src)
{
    static_assert(N == 4 || N == 8 || N == 16, "cp.async copies 4, 8 or 16 bytes");
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(smem_u32(dst)), "l"(src), "n"(N)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// 4-D tiled tensor copy global -> shared (coordinate x is innermost).
__device__ __forceinline__ void tensor4d_g2s(void *dst, const CUtensorMap *map, int x, int y, int z,
                                             int w, uint64_t *bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w),
                 "r"(smem_u32(bar)), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// --------------------------------------------- programmatic dependent launch

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --------------------------------------------------------- named barriers

__device__ __forceinline__ void named_bar_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------- thread-block clusters

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Hardware barrier over every thread of the cluster (all CTAs of a cluster are
// co-scheduled, so this cannot wait on a CTA that is not running).  Release /
// acquire: shared-memory writes before it are visible to remote reads after it.
// The cluster barriers here are the non-.aligned forms: a thread may reach them
// from code its warp entered divergently.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\t"
                 "barrier.cluster.wait.acquire;" ::: "memory");
}

// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void *local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    return r;
}

// Split cluster barrier: arrive (relaxed) early, wait later.  With
// fence_mbar_init() before the arrive, mbarriers initialized before it may be
// signalled by other CTAs of the cluster after the wait.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// Asynchronous stores into another CTA's shared memory (addresses from
// dsmem_addr): each counts its bytes on the mbarrier `bar` of the destination
// CTA (a shared::cluster address from dsmem_addr too), which completes its phase
// once the bytes it expects have all landed.
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];"
                 ::"r"(addr), "f"(v), "r"(bar)
                 : "memory");
}

// Stores into another CTA's shared memory (addresses from dsmem_addr); they are
// visible to that CTA after the next cluster barrier.
__device__ __forceinline__ void st_dsmem(uint32_t addr, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_dsmem_v4(uint32_t addr, float4 v)
{
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// Remote load without a memory clobber, so independent loads can be in flight
// together; being volatile it stays after cluster_sync() (also volatile).
__device__ __forceinline__ float ld_dsmem(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// ------------------------------------------------------------ tensor cores

// D = A * B + C, m16n8k16, A/B fp16, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1, const float (&c)[4])
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
                 : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]),
                   "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// D = A * B + C, m16n8k16, A/B bf16, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1, const float (&c)[4])
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
                 : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]),
                   "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2_trans(uint32_t &r0, uint32_t &r1, uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

// ------------------------------------------------------------- small math

// explicit shared-memory accesses (a pointer that went through integer
// alignment arithmetic no longer tells the compiler its address space)
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_bits_to_float(uint16_t v)
{
    return __uint_as_float((uint32_t)v << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

}  // namespace gattn
