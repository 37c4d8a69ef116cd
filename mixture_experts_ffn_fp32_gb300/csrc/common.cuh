// Device helpers shared by the kernels of libmoe: inline-PTX wrappers for
// mbarrier, TMA (cp.async.bulk.tensor) and the 5th-generation tensor core
// (tcgen05 + tensor memory), bounded waits, and BF16 packing.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MOE_DEV __device__ __forceinline__

// Bits of the device-side error word kept at the start of every workspace.
enum : int {
    ERRBIT_TIMEOUT = 1,  // a bounded wait ran out of time; the kernel stopped early
    ERRBIT_INDEX = 2,    // an expert id outside [0, E) was met and skipped
};

MOE_DEV uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MOE_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

MOE_DEV uint32_t lane_id() { return threadIdx.x & 31u; }

// Programmatic dependent launch: every kernel of the forward is launched with
// programmatic stream serialisation, so it may start while its predecessor in
// the stream is still running. pdl_wait() blocks until the predecessor grid
// has completed and its memory is visible; it must precede any read of the
// predecessor's outputs (and any write the predecessor might read).
// pdl_trigger() lets the next kernel in the stream begin launching.
MOE_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
MOE_DEV void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

MOE_DEV void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

MOE_DEV void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

MOE_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Acquire at cluster scope: for barriers a peer CTA of the cluster arrives on.
MOE_DEV bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---------------------------------------------------------------------------
// Thread-block clusters
// ---------------------------------------------------------------------------
MOE_DEV uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster; orders memory at cluster scope.
MOE_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// The shared::cluster address of the variable at shared::cta address `saddr`
// in the CTA of cluster rank `rank`.
MOE_DEV uint32_t map_shared_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// The two halves of cluster_sync, for work between the arrival and the wait.
MOE_DEV void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
MOE_DEV void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

// FP32 load from the shared memory of a CTA of the cluster (shared::cluster address).
MOE_DEV float ld_shared_cluster_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}

// Arrive on an mbarrier of another CTA of the cluster (shared::cluster address).
MOE_DEV void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

MOE_DEV void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

MOE_DEV void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared state of the bounded waits of one CTA.
struct WaitCtx {
    int* err;                // global error word
    volatile int* abort;     // shared flag: some wait of this CTA gave up
    uint64_t timeout_ns;
};

// Wait for the phase of `bar` with parity `parity` to complete. Gives up
// (returns false) when another wait of the CTA gave up, or after timeout_ns,
// in which case it raises the CTA's abort flag and the global error bit.
// cluster: acquire at cluster scope (a peer CTA arrives on `bar`).
MOE_DEV bool bounded_wait(uint32_t bar, uint32_t parity, const WaitCtx& w, bool cluster = false) {
    auto poll = [&] { return cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (poll()) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (poll()) return true;
        if (*w.abort) return false;
        if (globaltimer_ns() - t0 > w.timeout_ns) {
            *w.abort = 1;
            atomicOr(w.err, ERRBIT_TIMEOUT);
            return false;
        }
    }
}

// Global counters that CTAs of one launch release to each other: the writer
// orders its stores (generic proxy) before the async proxy and the counter,
// the reader acquires the counter and orders it before its tensor-map copies.
MOE_DEV void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

MOE_DEV unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

MOE_DEV void release_add_gpu(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid barrier without initial state (one-launch kernels whose CTAs are all
// resident): every CTA stores this launch's tag (grid_epoch_tag: unique per
// launch on a workspace, graph replays included) into its own tag with
// release order and waits until every tag carries it. Tags sit one per
// 128-byte line; the epoch word sits on line GRID_EPOCH_LINE.
constexpr int GRID_TAG_STRIDE = 16;  // 64-bit words between tags
constexpr int GRID_EPOCH_LINE = 256;  // the epoch word's line, after 256 CTAs' tag lines

MOE_DEV void st_release_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

MOE_DEV unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

MOE_DEV void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// The grid barrier's tag for this launch: one more than the epoch word that
// the previous launch on the same workspace left there (read after
// griddepcontrol.wait, so that launch has completed). Once every CTA has
// read the word - after the barrier - CTA 0 stores the new value back
// (grid_epoch_store), so each launch, eager or a replay of a captured graph
// (whose launch parameters never change), waits for tags no earlier launch
// wrote, and the tags need no zeroing.
MOE_DEV unsigned long long grid_epoch_tag(const unsigned long long* epoch) { return ld_relaxed_u64(epoch) + 1ull; }
MOE_DEV void grid_epoch_store(unsigned long long* epoch, unsigned long long tag) {
    if (blockIdx.x == 0 && threadIdx.x == 0) st_release_u64(epoch, tag);
}

// Called by every thread of each CTA once the CTA's tag was stored (ntags <=
// blockDim.x): thread i watches tag i (relaxed loads), the CTA combines the
// outcomes, and an acquire fence orders the tags seen before the loads that
// follow. False when timeout_ns ran out (the error word gets ERRBIT_TIMEOUT).
MOE_DEV bool grid_tags_wait_cta(const unsigned long long* tags, int ntags, unsigned long long gid,
                                uint64_t timeout_ns, int* err) {
    bool ok = true;
    if (static_cast<int>(threadIdx.x) < ntags) {
        const uint64_t start = globaltimer_ns();
        while (ld_relaxed_u64(tags + GRID_TAG_STRIDE * threadIdx.x) != gid) {
            if (globaltimer_ns() - start > timeout_ns) {
                ok = false;
                break;
            }
        }
    }
    ok = __syncthreads_and(ok) != 0;
    fence_acq_rel_gpu();
    if (!ok && threadIdx.x == 0) atomicOr(err, ERRBIT_TIMEOUT);
    return ok;
}

// Asynchronous copies global -> shared (cp.async; 16 bytes: both addresses
// 16-byte aligned, 4 bytes: 4-byte aligned), all completed by cp_async_wait_all
// in the issuing thread (a __syncthreads then publishes them to the CTA).
MOE_DEV void cp_async_16(void* sdst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sdst)), "l"(gsrc) : "memory");
}
MOE_DEV void cp_async_4(void* sdst, const void* gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(sdst)), "l"(gsrc) : "memory");
}
MOE_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Wait until *p >= target (bounded like bounded_wait).
MOE_DEV bool bounded_wait_count(const unsigned* p, unsigned target, const WaitCtx& w) {
    if (ld_acquire_gpu(p) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (ld_acquire_gpu(p) >= target) return true;
        if (*w.abort) return false;
        if (globaltimer_ns() - t0 > w.timeout_ns) {
            *w.abort = 1;
            atomicOr(w.err, ERRBIT_TIMEOUT);
            return false;
        }
    }
}

// Same, ignoring the abort flag (used to drain copies already in flight).
MOE_DEV bool bounded_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) {
            atomicOr(err, ERRBIT_TIMEOUT);
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// Untiled bulk copy global -> shared of `bytes` bytes, completing on an
// mbarrier: both addresses 16-byte aligned, bytes a multiple of 16.
// ---------------------------------------------------------------------------
MOE_DEV void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// ---------------------------------------------------------------------------
// TMA: tiled bulk tensor loads global -> shared, completing on an mbarrier.
// ---------------------------------------------------------------------------
MOE_DEV void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

MOE_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

MOE_DEV void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

MOE_DEV void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Row gather: four rows r0..r3 of the column box at c0 of a 2-D tensor map
// whose box is one row high; they land as four consecutive box rows at dst
// (swizzled by their shared-memory address like a tiled copy of 4 rows).
MOE_DEV void tma_gather4(uint32_t dst, const CUtensorMap* map, int c0, int r0, int r1, int r2, int r3,
                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
        : "memory");
}

// CTA-pair forms (.cta_group::2): the copy lands in this CTA's shared memory
// and completes its bytes on `bar`, a shared::cluster address that may name
// the barrier of the peer CTA (the even CTA's, which counts both halves).
MOE_DEV void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

MOE_DEV void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

MOE_DEV void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory allocation, MMA, commit, loads.
// ---------------------------------------------------------------------------
MOE_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}

MOE_DEV void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// The same three for a CTA pair (cta_group::2): one warp of each of the two
// CTAs executes each of them; both CTAs receive the same column address.
MOE_DEV void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}

MOE_DEV void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

MOE_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

MOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem], BF16 inputs, FP32 accumulation.
MOE_DEV void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// CTA-pair MMA (cta_group::2), issued by one thread of the even CTA: M = 256
// rows, A rows 0-127 and accumulator lanes from the even CTA, rows 128-255
// from the odd one; B's N columns split in halves, the first half in the
// even CTA's shared memory. Descriptors name the same offsets in both CTAs.
MOE_DEV void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Pair commits: arrive on `bar` (same offset) in every CTA of `cta_mask`, or
// in this CTA only, once this thread's tcgen05 operations have completed.
MOE_DEV void tc_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

MOE_DEV void tc_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far has completed.
MOE_DEV void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp receives
// row (lane base + i), columns [col, col + 16).
MOE_DEV void tc_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

MOE_DEV void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile whose
// base is 1024-byte aligned (descriptor version 1, swizzle mode 2 = 128 B).
//   K-major tile (rows of 64 BF16 along K): lbo unused (16), sbo = 1024
//   (distance between 8-row groups); advance the start by 32 B per 16-wide K step.
//   MN-major tile (rows of 64 BF16 along N, one row per k): lbo = distance
//   between 64-column strips, sbo = 1024 (distance between 8-k groups).
MOE_DEV uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16;
    d |= static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: FP32 accumulator, BF16 A
// and B, A K-major, B K-major (b_mn_major = 0) or MN-major (1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int b_mn_major) {
    return (1u << 4)                                  // D format: F32
           | (1u << 7)                                // A format: BF16
           | (1u << 10)                               // B format: BF16
           | (static_cast<uint32_t>(b_mn_major) << 16)  // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// ---------------------------------------------------------------------------
// BF16 helpers
// ---------------------------------------------------------------------------
MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

MOE_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
MOE_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// 24-bit storage of an FP32 value: rounded to nearest (ties to even) at 16
// significant bits and kept as the float's top 24 bits, returned as
// (hi16 << 8) | lo8. Infinities pass through, a NaN stays a NaN, a finite
// value that rounds past the largest float becomes an infinity (IEEE
// rounding). f24_to_f32 puts the 24 bits back exactly.
MOE_DEV uint32_t f32_to_f24(float v) {
    const uint32_t u = __float_as_uint(v);
    if ((u & 0x7F800000u) == 0x7F800000u) return (u >> 8) | ((u & 0x007FFFFFu) ? 0x4000u : 0u);
    return (u + 0x7Fu + ((u >> 8) & 1u)) >> 8;
}
MOE_DEV float f24_to_f32(uint32_t hi16, uint32_t lo8) { return __uint_as_float((hi16 << 16) | (lo8 << 8)); }

MOE_DEV float silu_f(float a) { return a / (1.0f + __expf(-a)); }
