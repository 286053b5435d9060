// Tensor-core rate probe: how many cycles one SM's tensor core takes per
// kind::f16 MMA (M = 128, N = 256, K = 16, FP16 x FP16 -> FP32) when one
// thread issues them back to back from shared memory, with no loads, no
// epilogue and no barrier waits in between.
//
// The roofline of "02_mixed_precision_gemm" README ("Experimental Setup")
// takes the dense tensor peak as MACs per SM per clock x SMs x 2 x clock.
// The pages give that figure for their own GPU only; this probe measures the
// per-SM factor on the device itself, so that
//     theoretical peak = SMs x (2 * 128 * 256 * 16 / cycles per MMA) x max clock
// rests on a measurement rather than on a data-sheet number. %clock64 counts
// SM cycles at whatever clock the SM runs, so the result does not depend on
// the clock during the probe.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace mpgemm {

// 48 KB of operands plus a barrier and the tensor-memory slot; the launch asks
// for more shared memory than half an SM holds, so each SM runs one probe CTA
// and its tensor core serves that CTA alone.
constexpr int kProbeOperandBytes = 49152;
constexpr int kProbeSmemBytes = 160 * 1024;

// One warp per CTA. out[2 * blockIdx.x] = cycles from the first MMA's issue
// to the completion of the last, out[2 * blockIdx.x + 1] = 1 if the final
// completion was seen within wait_limit_ns (0: the wait gave up).
__global__ void __launch_bounds__(32, 1)
    mma_rate_probe(int32_t mmas, uint64_t wait_limit_ns, unsigned long long* out) {
    extern __shared__ uint8_t probe_smem[];
    const uint32_t raw = ptx::smem_addr(probe_smem);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* g = probe_smem + (base - raw);
    const uint32_t sA = base, sB = base + 16384, bar = base + kProbeOperandBytes;
    uint32_t* slot = reinterpret_cast<uint32_t*>(g + kProbeOperandBytes + 16);
    const int lane = threadIdx.x;
    // zero operands: the values do not change an MMA's cycle count
    for (int i = lane; i < kProbeOperandBytes / 16; i += 32)
        reinterpret_cast<uint4*>(g)[i] = make_uint4(0u, 0u, 0u, 0u);
    ptx::fence_proxy_async_smem();
    if (lane == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_barrier_init();
    }
    ptx::tmem_alloc(ptx::smem_addr(slot), 256);
    ptx::tmem_relinquish();
    ptx::tc_fence_before_sync();
    __syncwarp();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *slot;
    if (lane == 0) {
        // A K-major (128 rows of 64 halves), B N-major (four 64-column boxes
        // of 8 KB): the descriptors of the GEMM kernel's one-CTA 128 x 256 tile
        const uint32_t idesc = ptx::idesc_f16_f32(128, 256, false, true);
        unsigned long long c0, c1;
        asm volatile("mov.u64 %0, %%clock64;" : "=l"(c0));
        for (int32_t i = 0; i < mmas; ++i) {
            const int kk = i & 3;
            ptx::mma_f16(tmem, ptx::smem_desc_sw128(sA + kk * 32, 16, 1024),
                         ptx::smem_desc_sw128(sB + kk * 2048, 8192, 1024), idesc, i > 0);
        }
        ptx::mma_commit(bar);
        bool ok = true;
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(bar, 0)) {
            if (ptx::globaltimer_ns() - t0 > wait_limit_ns) {
                ok = false;
                break;
            }
        }
        asm volatile("mov.u64 %0, %%clock64;" : "=l"(c1));
        out[2 * blockIdx.x] = c1 - c0;
        out[2 * blockIdx.x + 1] = ok ? 1ull : 0ull;
        if (!ok) {
            // let the MMAs still in flight finish (bounded) before the
            // tensor memory they write is released
            const uint64_t t1 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar, 0) && ptx::globaltimer_ns() - t1 < wait_limit_ns) {
            }
        }
    }
    ptx::tc_fence_before_sync();
    __syncwarp();
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, 256);
}

}  // namespace mpgemm
