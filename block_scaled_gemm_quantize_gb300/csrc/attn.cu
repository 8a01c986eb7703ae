// attn.cu -- FP8 attention over an FP8 KV cache on sm_103a (tcgen05 + TMA + TMEM).
//
// "NVIDIA NeMo RL logra una aceleracion del 48%..." (hotbookzone.com),
// "Ganancias de rendimiento en el mundo real": extending FP8 to the KV cache
// and the attention operations takes the speedup from the linear layers'
// 15-25 % to about 48 %; "El avance tecnico": attention otherwise stays in
// BF16.  Here both attention products run in FP8 on the tensor cores:
//   S = Q K^T  (Q one scale per token and head, 1x128; K one scale per 128
//               tokens and head, 128x128 -- the KV cache layout)
//   P = exp(S - running max)   in fp32, then E4M3 with the scale 1/448 (its
//               maximum is 1 by construction)
//   O = P V    (V per 128 tokens and head), rescaled online in fp32.
//
// One CTA per (128 query rows, head), 16 warps:
//   warp 0     TMA: the Q tile once, then K and V tiles of 128 keys into a
//              3-stage ring.
//   warp 1     TMEM owner and MMA issuer: S_j into one of two 128-column TMEM
//              buffers (4 x tcgen05.mma.kind::f8f6f4, K-major operands), and
//              O_j = P_j V_j into one of two more (P from shared memory,
//              K-major; V MN-major), issued one tile behind S so that the
//              softmax of tile j overlaps the MMAs of tile j+1.
//   warps 4-11 softmax, AT_SPLIT threads per query row (its TMEM lane; the
//              warps w, w + 4, ... of a lane quarter own consecutive
//              128/AT_SPLIT-column parts): one TMEM read of the thread's
//              scores, the row max exchanged among the row's threads through
//              shared memory and a bounded mbarrier, the tile's running-max
//              factor handed to the correction warps, then exp2, the partial
//              row sum and the E4M3 codes of 448 P written into the
//              128-byte-swizzled P buffer.
//   warps 12-15 O correction, one thread per query row: each tile's O partial
//              read from TMEM and folded into the row's 128 fp32 accumulators
//              with the running-max factor and the V tile's scale, off the
//              softmax warps' path.  At the end O / l is stored as bf16.
// Every wait is bounded; a role that gives up records the timeout in a
// status word read by fp8bs_device_status, and the CTA leaves after draining
// its own asynchronous work.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "attn_kernels.h"
#include "fp8_math.cuh"
#include "gemm_kernels.h"
#include "ptx_sm100.cuh"

namespace fp8bs {

__device__ int g_attn_status;   // 0 = ok, else a negative fp8bs status (bounded wait expired)

namespace {

constexpr int AT_ROWS = 128, AT_KEYS = 128, AT_D = 128;
constexpr int AT_STAGES = 3;
#ifndef FP8BS_ATTN_SPLIT
#define FP8BS_ATTN_SPLIT 2
#endif
// softmax threads per query row: each owns 128 / AT_SPLIT columns of S and O
constexpr int AT_SPLIT = FP8BS_ATTN_SPLIT;
constexpr int AT_CPT = 128 / AT_SPLIT;
constexpr int AT_SM_WARPS = 4 * AT_SPLIT;
constexpr int AT_SM_WARP0 = 4;                            // first softmax warp
constexpr int AT_CO_WARP0 = AT_SM_WARP0 + AT_SM_WARPS;    // first O-correction warp (4 of them)
constexpr int AT_THREADS = 128 + 32 * AT_SM_WARPS + 128;
// setmaxnreg split of the launch's registers (65536 / threads, in steps of 8):
// control warps, softmax warps, O-correction warps (128 fp32 accumulators)
constexpr int AT_REGS_LAUNCH = (65536 / AT_THREADS) & ~7;
constexpr int AT_REGS_LOW = 48;
constexpr int AT_REGS_CO = 176;
constexpr int AT_REGS_HIGH =
    ((AT_REGS_LAUNCH * AT_THREADS - 128 * AT_REGS_LOW - 128 * AT_REGS_CO) / (32 * AT_SM_WARPS)) & ~7;
static_assert(AT_REGS_HIGH <= 256 && AT_REGS_HIGH >= 128 &&
                  128 * AT_REGS_LOW + 32 * AT_SM_WARPS * AT_REGS_HIGH + 128 * AT_REGS_CO <=
                      AT_REGS_LAUNCH * AT_THREADS,
              "register split");
constexpr uint32_t AT_TILE = AT_ROWS * AT_D;          // 16 KiB of codes
constexpr uint32_t AT_Q_OFF = 0;
constexpr uint32_t AT_KV_OFF = AT_TILE;               // stage s: K at +0, V at +16 KiB
constexpr uint32_t AT_P_OFF = AT_KV_OFF + AT_STAGES * 2 * AT_TILE;
constexpr uint32_t AT_BAR_OFF = AT_P_OFF + 2 * AT_TILE;
// q_full, kv_full[3], kv_empty[3], s_full[2], s_empty[2], p_full[2], p_empty[2],
// o_full[2], o_empty[2], done, xchg[4], a_full[4], l_full
constexpr int AT_NUM_BARS = 1 + 2 * AT_STAGES + 6 * 2 + 1 + 4 + 5;
constexpr uint32_t AT_TMEMSLOT_OFF = AT_BAR_OFF + AT_NUM_BARS * 8;
// row-max / row-sum exchange among the threads of a row: [parity][part][row]
constexpr uint32_t AT_XCHG_OFF = (AT_TMEMSLOT_OFF + 16 + 15) & ~15u;
// running-max factors handed to the O-correction warps ([tile % 4][row]) and
// the final row sums ([row])
constexpr uint32_t AT_ALPHA_OFF = AT_XCHG_OFF + 2 * AT_SPLIT * 128 * 4;
constexpr uint32_t AT_L_OFF = AT_ALPHA_OFF + 4 * 128 * 4;
constexpr uint32_t AT_SMEM_BYTES = 1024 + AT_L_OFF + 128 * 4;
constexpr float AT_LOG2_448 = 8.807354922057604f;   // log2(448)
static_assert(AT_SMEM_BYTES <= 232448, "shared memory budget (attention)");
constexpr uint64_t AT_WAIT_NS = 4000000000ull;
constexpr uint64_t AT_DRAIN_NS = 200000000ull;

__device__ __forceinline__ bool at_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t n = 0;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++n & 63u) == 0 && global_timer_ns() - t0 > AT_WAIT_NS) {
            atomicExch(&g_attn_status, kStatusDeviceTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ bool at_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > AT_DRAIN_NS) return false;
    return true;
}

__device__ __forceinline__ void add_f32x2(uint64_t& acc, uint64_t b) {   // two fp32 adds, one instruction
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc) : "l"(b));
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Largest V tile scale of kv head g (over all its key tiles), reduced across
// the warp: P is scaled by sv_j / this maximum (at most 1) before it is
// quantized, so the products of every key tile accumulate in one unit.
__device__ __forceinline__ float head_max_sv(const float* sv, int64_t seq_k, int32_t hkv, int g, int lane) {
    const int64_t nt = (seq_k + 127) / 128;
    float m = 0.0f;
    for (int64_t t = lane; t < nt; t += 32) m = fmaxf(m, __ldg(sv + t * hkv + g));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    return m;
}

// number of 128-key tiles a CTA visits (0: no visible key for any of its rows)
__device__ __forceinline__ int kv_tiles(const AttnParams& p, int64_t q0) {
    const int64_t n_all = (p.seq_k + AT_KEYS - 1) / AT_KEYS;
    if (!p.causal) return static_cast<int>(n_all);
    const int64_t last_row = min(q0 + AT_ROWS - 1, p.seq_q - 1);
    const int64_t last_key = min(last_row + (p.seq_k - p.seq_q), p.seq_k - 1);
    if (last_key < 0) return 0;
    return static_cast<int>(min(n_all, last_key / AT_KEYS + 1));
}

__global__ void __launch_bounds__(AT_THREADS, 1)
    k_fp8_attn_fwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + AT_BAR_OFF;
    const uint32_t q_full = bars;
    auto kv_full = [&](int s) { return bars + 8u * (1 + s); };
    auto kv_empty = [&](int s) { return bars + 8u * (1 + AT_STAGES + s); };
    auto s_full = [&](int b) { return bars + 8u * (1 + 2 * AT_STAGES + b); };
    auto s_empty = [&](int b) { return bars + 8u * (3 + 2 * AT_STAGES + b); };
    auto p_full = [&](int b) { return bars + 8u * (5 + 2 * AT_STAGES + b); };
    auto p_empty = [&](int b) { return bars + 8u * (7 + 2 * AT_STAGES + b); };
    auto o_full = [&](int b) { return bars + 8u * (9 + 2 * AT_STAGES + b); };
    auto o_empty = [&](int b) { return bars + 8u * (11 + 2 * AT_STAGES + b); };
    const uint32_t done_bar = bars + 8u * (13 + 2 * AT_STAGES);
    auto xchg_bar = [&](int q) { return bars + 8u * (14 + 2 * AT_STAGES + q); };
    auto a_full = [&](int b) { return bars + 8u * (18 + 2 * AT_STAGES + b); };
    const uint32_t l_full = bars + 8u * (22 + 2 * AT_STAGES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + AT_TMEMSLOT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y;
    const int g = h / (p.hq / p.hkv);
    // causal: the last query tiles see the most keys, so they start first
    const int64_t q0 = static_cast<int64_t>(p.causal ? gridDim.x - 1 - blockIdx.x : blockIdx.x) * AT_ROWS;
    const int n = kv_tiles(p, q0);

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        mbar_init(q_full, 1);
        for (int s = 0; s < AT_STAGES; s++) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(s_full(b), 1);
            mbar_init(s_empty(b), AT_SM_WARPS);   // one arrival per softmax warp
            mbar_init(p_full(b), AT_SM_WARPS);
            mbar_init(p_empty(b), 1);
            mbar_init(o_full(b), 1);
            mbar_init(o_empty(b), 4);             // the O-correction warps
            mbar_init(a_full(b), AT_SM_WARPS);
            mbar_init(a_full(b + 2), AT_SM_WARPS);
        }
        mbar_init(l_full, AT_SM_WARPS);
        mbar_init(done_bar, 1);
        for (int q = 0; q < 4; q++) mbar_init(xchg_bar(q), 32 * AT_SPLIT);   // the warps of a lane quarter
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < AT_SM_WARP0) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(AT_REGS_LOW));
    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0 && n > 0) {
            bool ok = true;
            int issued = 0;
            mbar_arrive_expect_tx(q_full, AT_TILE);
            tma_load_2d(sbase + AT_Q_OFF, &tmQ, h * AT_D, static_cast<int32_t>(q0), q_full);
            for (int j = 0; j < n; j++) {
                const int s = j % AT_STAGES;
                if (!at_wait(kv_empty(s), ((j / AT_STAGES) & 1u) ^ 1u)) { ok = false; break; }
                const uint32_t dst = sbase + AT_KV_OFF + s * 2 * AT_TILE;
                mbar_arrive_expect_tx(kv_full(s), 2 * AT_TILE);
                tma_load_2d(dst, &tmK, g * AT_D, j * AT_KEYS, kv_full(s));
                tma_load_2d(dst + AT_TILE, &tmV, g * AT_D, j * AT_KEYS, kv_full(s));
                issued++;
            }
            at_drain(q_full, 0);   // the Q copy has landed before this thread leaves
            if (!ok) {
                for (int i = 0; i < AT_STAGES && i < issued; i++) {
                    const int j = issued - 1 - i;
                    at_drain(kv_full(j % AT_STAGES), (j / AT_STAGES) & 1u);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && n > 0) {
            bool ok = at_wait(q_full, 0), issued_mma = false;
            auto issue_s = [&](int j) -> bool {
                const int s = j % AT_STAGES, b = j & 1;
                if (!at_wait(kv_full(s), (j / AT_STAGES) & 1u)) return false;
                if (!at_wait(s_empty(b), ((j >> 1) & 1u) ^ 1u)) return false;
                tc_fence_after();
                const uint32_t kS = sbase + AT_KV_OFF + s * 2 * AT_TILE;
#pragma unroll
                for (int k4 = 0; k4 < AT_D / 32; k4++)
                    mma_f8f6f4(tmem + b * 128, smem_desc_sw128(sbase + AT_Q_OFF + k4 * 32, 16, 1024),
                               smem_desc_sw128(kS + k4 * 32, 16, 1024), p.idesc_s, k4 > 0 ? 1u : 0u);
                issued_mma = true;
                mma_commit(s_full(b));
                return true;
            };
            auto issue_o = [&](int j) -> bool {
                const int s = j % AT_STAGES, b = j & 1;
                if (!at_wait(p_full(b), (j >> 1) & 1u)) return false;
                if (!at_wait(o_empty(b), ((j >> 1) & 1u) ^ 1u)) return false;
                tc_fence_after();
                const uint32_t vS = sbase + AT_KV_OFF + s * 2 * AT_TILE + AT_TILE;
                const uint32_t pS = sbase + AT_P_OFF + b * AT_TILE;
#pragma unroll
                for (int k4 = 0; k4 < AT_KEYS / 32; k4++)
                    // P: K-major (keys contiguous in a row); V: MN-major, one
                    // 128-wide atom, 32 keys x 128 B further per K step
                    mma_f8f6f4(tmem + 256 + b * 128, smem_desc_sw128(pS + k4 * 32, 16, 1024),
                               smem_desc_sw128(vS + k4 * 4096, 1024, 1024), p.idesc_o, k4 > 0 ? 1u : 0u);
                mma_commit(o_full(b));
                mma_commit(p_empty(b));
                mma_commit(kv_empty(s));
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; ok && j < n; j++) {
                if (j + 1 < n && !issue_s(j + 1)) { ok = false; break; }
                if (!issue_o(j)) { ok = false; break; }
            }
            if (!ok && issued_mma) {
                mma_commit(done_bar);
                at_drain(done_bar, 0);
            }
        }
    } else if (warp >= AT_SM_WARP0 && warp < AT_CO_WARP0) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(AT_REGS_HIGH));
        // -------------------------------------------------------- softmax
        const int quarter = warp & 3;
        const int cq = (warp - AT_SM_WARP0) >> 2;                 // column part: AT_CPT cq ..
        const int r = quarter * 32 + lane;                       // TMEM lane = query row in the tile
        const int64_t row = q0 + r;
        const bool row_ok = row < p.seq_q;
        const int64_t crow = row_ok ? row : p.seq_q - 1;
        const int64_t offs = p.seq_k - p.seq_q;
        const int64_t last_key = p.causal ? min(crow + offs, p.seq_k - 1) : p.seq_k - 1;
        // keys every row of this CTA sees: a tile below this needs no mask
        const int64_t all_vis = p.causal ? min(q0 + offs, p.seq_k - 1) : p.seq_k - 1;
        const float qs = __ldg(p.sq + static_cast<int64_t>(h) * p.seq_q + crow);
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t col_off = static_cast<uint32_t>(cq * AT_CPT);
        const uint32_t xbuf = sbase + AT_XCHG_OFF;
        uint32_t xc = 0;                                          // exchanges done (parity)
        // combine v over the row's AT_SPLIT threads (max or sum); false on timeout
        auto exchange = [&](float& v, bool take_max) -> bool {
            const uint32_t par = xc & 1u;
            st_shared_f32(xbuf + ((par * AT_SPLIT + cq) * 128 + r) * 4, v);
            mbar_arrive(xchg_bar(quarter));
            if (!__all_sync(0xFFFFFFFFu, at_wait(xchg_bar(quarter), par))) return false;
            float t = take_max ? -INFINITY : 0.0f;
#pragma unroll
            for (int k = 0; k < AT_SPLIT; k++) {
                const float o = ld_shared_f32(xbuf + ((par * AT_SPLIT + k) * 128 + r) * 4);
                t = take_max ? fmaxf(t, o) : t + o;
            }
            v = t;
            xc++;
            return true;
        };
        float m = -INFINITY, l = 0.0f;   // l: this part's sum of 448 P (same max for all parts)
        bool ok = true;

        // K tile scales: lane i holds that of tile 32 w + i while the loop is
        // in window w (reloaded every 32 tiles) and a tile's is taken by a
        // shuffle.  A global load issued every tile would hold up the warp's
        // next TMEM-load wait until it lands.
        auto ksc = [&](int t) { return t < n ? __ldg(p.sk + static_cast<int64_t>(t) * p.hkv + g) : 0.0f; };
        float skw = 0.0f;
        for (int j = 0; ok && j < n; j++) {
            const int b = j & 1;
            if ((j & 31) == 0) skw = ksc(j + lane);
            const float sk_j = __shfl_sync(0xFFFFFFFFu, skw, j & 31);
            ok = __all_sync(0xFFFFFFFFu, at_wait(s_full(b), (j >> 1) & 1u));
            if (!ok) break;
            tc_fence_after();
            const bool full = static_cast<int64_t>(j) * AT_KEYS + AT_KEYS - 1 <= all_vis;   // CTA-uniform
            uint32_t sr[AT_CPT / 32][32];
            float lm[AT_CPT / 32];   // per-load maxima (fully visible tiles)
            if (full) {
#pragma unroll
                for (int u = 0; u < AT_CPT / 32; u++)
                    tmem_ld_max_32x32b_x32(tmem + lane_off + b * 128 + col_off + u * 32, sr[u], lm[u]);
            } else {
#pragma unroll
                for (int u = 0; u < AT_CPT / 32; u++)
                    tmem_ld_32x32b_x32(tmem + lane_off + b * 128 + col_off + u * 32, sr[u]);
            }
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_empty(b));   // S buffer read: hand it back
            const float c = qs * sk_j * p.scale_log2;
            const int64_t key0 = static_cast<int64_t>(j) * AT_KEYS + col_off;
            // scores in log2 units are raw * c with c > 0, so the row max is
            // max(raw) * c; masked keys become -inf.  Eight independent
            // partial maxima / sums keep the dependency chains short.
            float tm[8];
#pragma unroll
            for (int i = 0; i < 8; i++) tm[i] = -INFINITY;
            if (full) {   // every key of the tile is visible: the loads reduced the maxima
#pragma unroll
                for (int u = 0; u < AT_CPT / 32; u++) tm[u] = lm[u];
            } else {      // keys e <= lim are visible to this row
                const int lim = static_cast<int>(max(min(last_key - key0, static_cast<int64_t>(AT_CPT)),
                                                     static_cast<int64_t>(-1)));
#pragma unroll
                for (int e = 0; e < AT_CPT; e++) {
                    const float v = e <= lim ? __uint_as_float(sr[e >> 5][e & 31]) : -INFINITY;
                    sr[e >> 5][e & 31] = __float_as_uint(v);
                    tm[e & 7] = fmaxf(tm[e & 7], v);
                }
            }
            float tmax = fmaxf(fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3])),
                               fmaxf(fmaxf(tm[4], tm[5]), fmaxf(tm[6], tm[7])));
            tmax = tmax == -INFINITY ? -INFINITY : tmax * c;
            ok = exchange(tmax, true);
            if (!ok) break;
            const float m_new = fmaxf(m, tmax);
            const float alpha = m_new == -INFINITY ? 1.0f : ex2(m - m_new);
            const float shift = AT_LOG2_448 - (m_new == -INFINITY ? 0.0f : m_new);
            ok = __all_sync(0xFFFFFFFFu, at_wait(p_empty(b), ((j >> 1) & 1u) ^ 1u));
            if (!ok) break;
            // hand this tile's running-max factor to the O-correction warps, in
            // slot j % 4.  That slot's previous factor (tile j - 4) has been
            // read: P_j's buffer is free, so O_{j-2} = P_{j-2} V was issued, which
            // waited for the correction warps to drain O_{j-4}, and they read a
            // tile's factor before draining its O.
            if (cq == 0) st_shared_f32(sbase + AT_ALPHA_OFF + ((j & 3) * 128 + r) * 4, alpha);
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full(j & 3));
            // 448 P = 2^(raw c - m_new + log2 448) (masked: 2^-inf = 0), row sum, codes
            const uint32_t prow = sbase + AT_P_OFF + b * AT_TILE + r * 128;
            float rs[8];
#pragma unroll
            for (int i = 0; i < 8; i++) rs[i] = 0.0f;
#pragma unroll
            for (int ch = 0; ch < AT_CPT / 16; ch++) {            // 16 keys = one 16-byte chunk
                float pv[16];
#pragma unroll
                for (int e = 0; e < 16; e++) {
                    const int k = ch * 16 + e;
                    pv[e] = ex2(fmaf(__uint_as_float(sr[k >> 5][k & 31]), c, shift));
                    rs[e & 7] += pv[e];
                }
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; i++)
                    w[i] = cvt4_e4m3(pv[4 * i], pv[4 * i + 1], pv[4 * i + 2], pv[4 * i + 3]);
                const uint32_t cc = col_off / 16 + static_cast<uint32_t>(ch);
                st_shared_v4(prow + ((cc ^ (static_cast<uint32_t>(r) & 7u)) << 4), w[0], w[1], w[2], w[3]);
            }
            const float rsum = ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(b));
            l = l * alpha + rsum;
            m = m_new;
        }
        if (ok && n > 0) ok = exchange(l, false);                 // row sum over all parts
        // the row sum for the O-correction warps (always handed over, so that
        // they never wait for it in vain; a timeout above is already recorded)
        if (cq == 0) st_shared_f32(sbase + AT_L_OFF + r * 4, ok ? l : 0.0f);
        __syncwarp();
        if (lane == 0) mbar_arrive(l_full);
    } else if (warp >= AT_CO_WARP0) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(AT_REGS_CO));
        // ---------------------------------------------------- O correction
        // One thread per query row holds the row's 128 O columns in fp32:
        // per tile, acc = acc * alpha_t + (P_t V_t) * sv_t, with P_t V_t read
        // from TMEM and alpha_t from the softmax warps; at the end O / l.
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int64_t row = q0 + r;
        const bool row_ok = row < p.seq_q;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        uint64_t acc[64];   // the row's O columns as packed pairs
#pragma unroll
        for (int i = 0; i < 64; i++) acc[i] = 0;
        bool ok = true;
        auto vsc = [&](int t) { return t < n ? __ldg(p.sv + static_cast<int64_t>(t) * p.hkv + g) : 0.0f; };
        float svw = 0.0f;   // V scales: a window of 32 tiles across the lanes (as for K)
        for (int j = 0; ok && j < n; j++) {
            const int b = j & 1;
            if ((j & 31) == 0) svw = vsc(j + lane);
            const float sv_j = __shfl_sync(0xFFFFFFFFu, svw, j & 31);
            ok = __all_sync(0xFFFFFFFFu, at_wait(a_full(j & 3), (j >> 2) & 1u));
            if (!ok) break;
            const float alpha = ld_shared_f32(sbase + AT_ALPHA_OFF + ((j & 3) * 128 + r) * 4);
            ok = __all_sync(0xFFFFFFFFu, at_wait(o_full(b), (j >> 1) & 1u));
            if (!ok) break;
            tc_fence_after();
            const uint64_t a2 = pack_f32x2(__float_as_uint(alpha), __float_as_uint(alpha));
            const uint64_t v2 = pack_f32x2(__float_as_uint(sv_j), __float_as_uint(sv_j));
#pragma unroll
            for (int u = 0; u < 4; u++) {
                uint32_t rr[32];
                tmem_ld_32x32b_x32(tmem + lane_off + 256 + b * 128 + u * 32, rr);
                tmem_wait_ld();
                if (u == 3) {   // last read of this O partial: hand the buffer back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(o_empty(b));
                }
#pragma unroll
                for (int q = 0; q < 16; q++) {
                    const uint64_t pv = mul_f32x2(pack_f32x2(rr[2 * q], rr[2 * q + 1]), v2);
                    uint64_t a = acc[u * 16 + q];
                    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(acc[u * 16 + q]) : "l"(a), "l"(a2), "l"(pv));
                }
            }
        }
        // O = sum(448 P * V * sv) / sum(448 P)
        if (ok) ok = __all_sync(0xFFFFFFFFu, at_wait(l_full, 0));
        if (ok && row_ok) {
            const float l = ld_shared_f32(sbase + AT_L_OFF + r * 4);
            const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
            uint16_t* o = reinterpret_cast<uint16_t*>(p.o) + row * p.ldo + static_cast<int64_t>(h) * AT_D;
#pragma unroll
            for (int c8 = 0; c8 < AT_D / 8; c8++) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const float2 f = unpack_f32x2(acc[c8 * 4 + i]);
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(f.x * inv_l, f.y * inv_l);
                    w[i] = *reinterpret_cast<uint32_t*>(&h2);
                }
                *reinterpret_cast<uint4*>(o + c8 * 8) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}


// ================================================================ two tiles
// Version 2: a CTA takes TWO 128-query tiles (A: rows q0.., B: rows
// q0 + 128..) of one head, which share every K/V tile, and keeps each
// tile's O accumulating in tensor memory:
//   TMEM columns   S_A 0-127, S_B 128-255, O_A 256-383, O_B 384-511.
//   warp 0         TMA: Q_A and Q_B once, K/V 128-key tiles into 3 stages.
//   warps 1, 2     MMA, one issuer per query tile: S_X(j) = Q_X K_j^T as soon
//                  as tile X's softmax has read S_X(j-1); O_X += P_X(j) V_j once
//                  P_X(j) is written and O_X has been rescaled for tile j.  The
//                  two tiles progress independently, so the tensor core works
//                  on one while the other is in softmax.
//   warps 4-7      softmax of tile A, warps 8-11 of tile B: one thread per
//                  query row holds the row's 128 scores (no exchange between
//                  threads), the row max (reduced by the TMEM loads on fully
//                  visible tiles), exp2, the row sum and the E4M3 codes of
//                  448 P (sv_j / svm) into a double-buffered, 128-byte-swizzled
//                  P buffer, svm the head's largest V tile scale: the factor
//                  is a shift of the exponent, so every tile's P V product
//                  lands in O_X in the unit of svm, and the row sum takes P
//                  unscaled.
//   warps 12-15    O correction, one thread per row of both tiles: before
//                  O_X(j) accumulates, O_X *= alpha_j (the running-max factor),
//                  read from and written back to TMEM -- only when a row of
//                  the warp changed its maximum; at the end O = O_X svm / l in
//                  bf16.
constexpr int A2_THREADS = 512;
constexpr uint32_t A2_Q_OFF = 0;                                  // Q_A, Q_B
constexpr uint32_t A2_KV_OFF = 2 * AT_TILE;                       // stage s: K +0, V +16 KiB
constexpr uint32_t A2_P_OFF = A2_KV_OFF + AT_STAGES * 2 * AT_TILE;  // P[X][b]
constexpr uint32_t A2_BAR_OFF = A2_P_OFF + 4 * AT_TILE;
// q_full, kv_full[3], kv_empty[3], s_full[2], s_empty[2], p_full[2][2],
// p_empty[2][2], o_done[2], corr_done[2], a_full[2][4], l_full[2], done[2]
constexpr int A2_NUM_BARS = 1 + 2 * AT_STAGES + 2 + 2 + 4 + 4 + 2 + 2 + 8 + 2 + 2;
constexpr uint32_t A2_TMEMSLOT_OFF = A2_BAR_OFF + A2_NUM_BARS * 8;
constexpr uint32_t A2_ALPHA_OFF = (A2_TMEMSLOT_OFF + 16 + 15) & ~15u;   // [X][4][128] fp32
constexpr uint32_t A2_L_OFF = A2_ALPHA_OFF + 2 * 4 * 128 * 4;           // [X][128] fp32
constexpr uint32_t A2_SMEM_BYTES = 1024 + A2_L_OFF + 2 * 128 * 4;
static_assert(A2_SMEM_BYTES <= 232448, "shared memory budget (attention, two tiles)");
// registers: 128 / thread at launch; control warps 48 and correction warps
// 80 (both decreases), softmax 192 (an increase, 128 scores per row):
// 128 * 48 + 256 * 192 + 128 * 80 == 512 * 128
constexpr int A2_REGS_LOW = 48, A2_REGS_SM = 192, A2_REGS_CO = 80;
static_assert(128 * A2_REGS_LOW + 256 * A2_REGS_SM + 128 * A2_REGS_CO == 512 * 128, "register split");
static_assert(A2_REGS_LOW <= 128 && A2_REGS_CO <= 128 && A2_REGS_SM >= 128, "setmaxnreg directions");

__global__ void __launch_bounds__(A2_THREADS, 1)
    k_fp8_attn_fwd2(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + A2_BAR_OFF;
    const uint32_t q_full = bars;
    auto kv_full = [&](int s) { return bars + 8u * (1 + s); };
    auto kv_empty = [&](int s) { return bars + 8u * (1 + AT_STAGES + s); };
    constexpr int B0 = 1 + 2 * AT_STAGES;
    auto s_full = [&](int x) { return bars + 8u * (B0 + x); };
    auto s_empty = [&](int x) { return bars + 8u * (B0 + 2 + x); };
    auto p_full = [&](int x, int b) { return bars + 8u * (B0 + 4 + 2 * x + b); };
    auto p_empty = [&](int x, int b) { return bars + 8u * (B0 + 8 + 2 * x + b); };
    auto o_done = [&](int x) { return bars + 8u * (B0 + 12 + x); };
    auto corr_done = [&](int x) { return bars + 8u * (B0 + 14 + x); };
    auto a_full = [&](int x, int k) { return bars + 8u * (B0 + 16 + 4 * x + k); };
    auto l_full = [&](int x) { return bars + 8u * (B0 + 24 + x); };
    auto done_bar = [&](int x) { return bars + 8u * (B0 + 26 + x); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + A2_TMEMSLOT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y;
    const int g = h / (p.hq / p.hkv);
    // causal: the last query tiles see the most keys, so they start first
    const int64_t q0 = static_cast<int64_t>(p.causal ? gridDim.x - 1 - blockIdx.x : blockIdx.x) * (2 * AT_ROWS);
    const int nA = q0 < p.seq_q ? kv_tiles(p, q0) : 0;
    const int nB = q0 + AT_ROWS < p.seq_q ? kv_tiles(p, q0 + AT_ROWS) : 0;
    const int n = max(nA, nB);

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        mbar_init(q_full, 1);
        for (int s = 0; s < AT_STAGES; s++) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 2);            // both MMA issuers
        }
        for (int x = 0; x < 2; x++) {
            mbar_init(s_full(x), 1);
            mbar_init(s_empty(x), 4);            // the tile's four softmax warps
            for (int b = 0; b < 2; b++) {
                mbar_init(p_full(x, b), 4);
                mbar_init(p_empty(x, b), 1);
            }
            mbar_init(o_done(x), 1);
            mbar_init(corr_done(x), 4);          // the four correction warps
            for (int k = 0; k < 4; k++) mbar_init(a_full(x, k), 4);
            mbar_init(l_full(x), 4);
            mbar_init(done_bar(x), 1);
        }
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(A2_REGS_LOW));
        if (warp == 0 && lane == 0 && n > 0) {
            // ---------------------------------------------------------- TMA
            bool ok = true;
            int issued = 0;
            mbar_arrive_expect_tx(q_full, 2 * AT_TILE);
            tma_load_2d(sbase + A2_Q_OFF, &tmQ, h * AT_D, static_cast<int32_t>(q0), q_full);
            tma_load_2d(sbase + A2_Q_OFF + AT_TILE, &tmQ, h * AT_D, static_cast<int32_t>(q0 + AT_ROWS), q_full);
            for (int j = 0; j < n; j++) {
                const int s = j % AT_STAGES;
                if (!at_wait(kv_empty(s), ((j / AT_STAGES) & 1u) ^ 1u)) { ok = false; break; }
                const uint32_t dst = sbase + A2_KV_OFF + s * 2 * AT_TILE;
                mbar_arrive_expect_tx(kv_full(s), 2 * AT_TILE);
                tma_load_2d(dst, &tmK, g * AT_D, j * AT_KEYS, kv_full(s));
                tma_load_2d(dst + AT_TILE, &tmV, g * AT_D, j * AT_KEYS, kv_full(s));
                issued++;
            }
            at_drain(q_full, 0);
            if (!ok) {
                for (int i = 0; i < AT_STAGES && i < issued; i++) {
                    const int j = issued - 1 - i;
                    at_drain(kv_full(j % AT_STAGES), (j / AT_STAGES) & 1u);
                }
            }
        } else if ((warp == 1 || warp == 2) && lane == 0 && n > 0) {
            // ------------------------------------------ MMA, one issuer per tile
            // warp 1 issues tile A's products, warp 2 tile B's, so that one
            // tile's softmax never waits behind the other's: S_X(j + 1) as soon
            // as the softmax has read S_X(j), O_X += P_X(j) V_j once P_X(j) is
            // written and O_X rescaled.  Both release each K/V stage; for the
            // key tiles past its own the issuer waits for the stage to fill
            // first, so that its release counts for that tile.
            const int x = warp - 1;
            const int nx = x ? nB : nA;
            bool ok = at_wait(q_full, 0), issued_mma = false;
            auto issue_s = [&](int j) -> bool {
                const int s = j % AT_STAGES;
                if (!at_wait(kv_full(s), (j / AT_STAGES) & 1u)) return false;
                if (j > 0 && !at_wait(s_empty(x), (j - 1) & 1u)) return false;   // S_X(j-1) was read
                tc_fence_after();
                const uint32_t kS = sbase + A2_KV_OFF + s * 2 * AT_TILE;
                const uint32_t qS = sbase + A2_Q_OFF + x * AT_TILE;
#pragma unroll
                for (int k4 = 0; k4 < AT_D / 32; k4++)
                    mma_f8f6f4(tmem + x * 128, smem_desc_sw128(qS + k4 * 32, 16, 1024),
                               smem_desc_sw128(kS + k4 * 32, 16, 1024), p.idesc_s, k4 > 0 ? 1u : 0u);
                issued_mma = true;
                mma_commit(s_full(x));
                return true;
            };
            auto issue_o = [&](int j) -> bool {
                const int s = j % AT_STAGES, b = j & 1;
                if (!at_wait(p_full(x, b), (j >> 1) & 1u)) return false;
                if (!at_wait(corr_done(x), j & 1u)) return false;                 // O_X rescaled for j
                tc_fence_after();
                const uint32_t vS = sbase + A2_KV_OFF + s * 2 * AT_TILE + AT_TILE;
                const uint32_t pS = sbase + A2_P_OFF + (2 * x + b) * AT_TILE;
#pragma unroll
                for (int k4 = 0; k4 < AT_KEYS / 32; k4++)
                    // P: K-major (keys contiguous in a row); V: MN-major, one
                    // 128-wide atom, 32 keys x 128 B further per K step
                    mma_f8f6f4(tmem + 256 + x * 128, smem_desc_sw128(pS + k4 * 32, 16, 1024),
                               smem_desc_sw128(vS + k4 * 4096, 1024, 1024), p.idesc_o,
                               (j > 0 || k4 > 0) ? 1u : 0u);
                mma_commit(o_done(x));
                mma_commit(p_empty(x, b));
                return true;
            };
            if (ok && nx > 0) ok = issue_s(0);
            for (int j = 0; ok && j < n; j++) {
                if (j < nx) {
                    if (j + 1 < nx && !issue_s(j + 1)) { ok = false; break; }
                    if (!issue_o(j)) { ok = false; break; }
                } else if (!at_wait(kv_full(j % AT_STAGES), (j / AT_STAGES) & 1u)) {
                    ok = false;
                    break;
                }
                mma_commit(kv_empty(j % AT_STAGES));
            }
            if (!ok && issued_mma) {
                mma_commit(done_bar(x));
                at_drain(done_bar(x), 0);
            }
        }
    } else if (warp < 12) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(A2_REGS_SM));
        // -------------------------------------------------------- softmax
        const int x = (warp - 4) >> 2;                  // query tile
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;              // TMEM lane = query row in the tile
        const int64_t tq0 = q0 + x * AT_ROWS;
        const int64_t row = tq0 + r;
        const bool row_ok = row < p.seq_q;
        const int64_t crow = row_ok ? row : p.seq_q - 1;
        const int nx = x ? nB : nA;
        const int64_t offs = p.seq_k - p.seq_q;
        const int64_t last_key = p.causal ? min(crow + offs, p.seq_k - 1) : p.seq_k - 1;
        // keys every row of this tile sees: a K/V tile below this needs no mask
        const int64_t all_vis = p.causal ? min(tq0 + offs, p.seq_k - 1) : p.seq_k - 1;
        const float qs = nx > 0 ? __ldg(p.sq + static_cast<int64_t>(h) * p.seq_q + crow) : 0.0f;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        float m = -INFINITY, l = 0.0f;   // l: the row's sum of 448 P
        bool ok = true;
        auto ksc = [&](int t) { return t < nx ? __ldg(p.sk + static_cast<int64_t>(t) * p.hkv + g) : 0.0f; };
        auto vsc = [&](int t) { return t < nx ? __ldg(p.sv + static_cast<int64_t>(t) * p.hkv + g) : 0.0f; };
        const float svm = head_max_sv(p.sv, p.seq_k, p.hkv, g, lane);
        const float lg_svm = svm > 0.0f ? lg2(svm) : 0.0f;
        float skw = 0.0f, svw = 0.0f;   // K / V tile scales: lane i holds tile 32 w + i of window w
        for (int j = 0; ok && j < nx; j++) {
            const int b = j & 1;
            if ((j & 31) == 0) {
                skw = ksc(j + lane);
                svw = vsc(j + lane);
            }
            const float sk_j = __shfl_sync(0xFFFFFFFFu, skw, j & 31);
            const float sv_j = __shfl_sync(0xFFFFFFFFu, svw, j & 31);
            // P of this tile scaled by sv_j / svm = 2^lv (a shift of the
            // exponent); its row sum is taken back by 2^-lv.  lv >= -60: a
            // zero (or smaller) scale still gives zero codes (448 P 2^-60 is
            // below half the least E4M3 subnormal) and an exact fp32 row sum.
            const float lv = fmaxf(lg2(sv_j) - lg_svm, -60.0f);
            const float inv_lv = ex2(-lv);
            ok = __all_sync(0xFFFFFFFFu, at_wait(s_full(x), j & 1u));
            if (!ok) break;
            tc_fence_after();
            const bool full = static_cast<int64_t>(j) * AT_KEYS + AT_KEYS - 1 <= all_vis;   // tile-uniform
            uint32_t sr[4][32];
            float lm[4];
            if (full) {
#pragma unroll
                for (int u = 0; u < 4; u++) tmem_ld_max_32x32b_x32(tmem + lane_off + x * 128 + u * 32, sr[u], lm[u]);
            } else {
#pragma unroll
                for (int u = 0; u < 4; u++) tmem_ld_32x32b_x32(tmem + lane_off + x * 128 + u * 32, sr[u]);
            }
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_empty(x));   // S_X read: the next S_X may be computed
            const float c = qs * sk_j * p.scale_log2;
            float tm[4];
            if (full) {
#pragma unroll
                for (int u = 0; u < 4; u++) tm[u] = lm[u];
            } else {   // keys e <= lim are visible to this row
                const int lim = static_cast<int>(max(min(last_key - static_cast<int64_t>(j) * AT_KEYS,
                                                         static_cast<int64_t>(AT_KEYS)), static_cast<int64_t>(-1)));
#pragma unroll
                for (int u = 0; u < 4; u++) tm[u] = -INFINITY;
#pragma unroll
                for (int e = 0; e < AT_KEYS; e++) {
                    const float v = e <= lim ? __uint_as_float(sr[e >> 5][e & 31]) : -INFINITY;
                    sr[e >> 5][e & 31] = __float_as_uint(v);
                    tm[e >> 5] = fmaxf(tm[e >> 5], v);
                }
            }
            float tmax = fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3]));
            tmax = tmax == -INFINITY ? -INFINITY : tmax * c;
            const float m_new = fmaxf(m, tmax);
            const float alpha = (m_new == -INFINITY || m_new == m) ? 1.0f : ex2(m - m_new);
            const float shift = AT_LOG2_448 + lv - (m_new == -INFINITY ? 0.0f : m_new);
            // P_X's buffer b is free once O_X(j - 2) has completed
            ok = __all_sync(0xFFFFFFFFu, at_wait(p_empty(x, b), ((j >> 1) & 1u) ^ 1u));
            if (!ok) break;
            // the running-max factor for the correction warps, slot j % 4 (its
            // previous value, tile j - 4, was read before O_X(j - 2) was issued)
            st_shared_f32(sbase + A2_ALPHA_OFF + ((x * 4 + (j & 3)) * 128 + r) * 4, alpha);
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full(x, j & 3));
            // 448 P = 2^(raw c - m_new + log2 448) (masked: 0), row sum, codes;
            // the argument and the row sum in packed pairs (f32x2)
            const uint32_t prow = sbase + A2_P_OFF + (2 * x + b) * AT_TILE + r * 128;
            const uint64_t c2 = pack_f32x2(__float_as_uint(c), __float_as_uint(c));
            const uint64_t sh2 = pack_f32x2(__float_as_uint(shift), __float_as_uint(shift));
            uint64_t rs[4];
#pragma unroll
            for (int i = 0; i < 4; i++) rs[i] = 0;
#pragma unroll
            for (int ch = 0; ch < AT_KEYS / 16; ch++) {          // 16 keys = one 16-byte chunk
                float pv[16];
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    const int k = ch * 16 + e;
                    uint64_t a2 = sh2;
                    fma_f32x2(a2, pack_f32x2(sr[k >> 5][k & 31], sr[k >> 5][(k & 31) + 1]), c2);
                    const float2 a = unpack_f32x2(a2);
                    pv[e] = ex2(a.x);
                    pv[e + 1] = ex2(a.y);
                    add_f32x2(rs[(e >> 1) & 3], pack_f32x2(__float_as_uint(pv[e]), __float_as_uint(pv[e + 1])));
                }
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; i++) w[i] = cvt4_e4m3(pv[4 * i], pv[4 * i + 1], pv[4 * i + 2], pv[4 * i + 3]);
                st_shared_v4(prow + ((static_cast<uint32_t>(ch) ^ (static_cast<uint32_t>(r) & 7u)) << 4), w[0], w[1],
                             w[2], w[3]);
            }
            float2 q0 = unpack_f32x2(rs[0]), q1 = unpack_f32x2(rs[1]), q2 = unpack_f32x2(rs[2]), q3 = unpack_f32x2(rs[3]);
            const float rsum = (((q0.x + q1.x) + (q2.x + q3.x)) + ((q0.y + q1.y) + (q2.y + q3.y))) * inv_lv;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(x, b));
            l = l * alpha + rsum;
            m = m_new;
        }
        // the row sum for the correction warps (always handed over, so that
        // they never wait for it in vain; a timeout above is already recorded)
        st_shared_f32(sbase + A2_L_OFF + (x * 128 + r) * 4, ok ? l : 0.0f);
        __syncwarp();
        if (lane == 0) mbar_arrive(l_full(x));
    } else {
        // (80 is below the launch's 128: a decrease)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(A2_REGS_CO));
        // ------------------------------------------------- O correction
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        bool ok = true;
        const float svm = head_max_sv(p.sv, p.seq_k, p.hkv, g, lane);
        for (int j = 0; ok && j < n; j++) {
#pragma unroll
            for (int x = 0; x < 2; x++) {
                if (j >= (x ? nB : nA)) continue;
                ok = __all_sync(0xFFFFFFFFu, at_wait(a_full(x, j & 3), (j >> 2) & 1u));
                if (!ok) break;
                // O_X holds its sum in the unit of the largest V scale, so only
                // the running-max factor rescales it; while no row of this warp
                // changed its maximum, O_X(j) may follow O_X(j - 1) unwaited (the
                // products of one accumulator run in order)
                const float f = ld_shared_f32(sbase + A2_ALPHA_OFF + ((x * 4 + (j & 3)) * 128 + r) * 4);
                if (j > 0 && __any_sync(0xFFFFFFFFu, f != 1.0f)) {
                    ok = __all_sync(0xFFFFFFFFu, at_wait(o_done(x), (j - 1) & 1u));   // O_X(j-1) complete
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t f2 = pack_f32x2(__float_as_uint(f), __float_as_uint(f));
                    const uint32_t ta = tmem + lane_off + 256 + x * 128;
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        uint32_t rr[32];
                        tmem_ld_32x32b_x32(ta + u * 32, rr);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 16; q++) {
                            const uint64_t v = mul_f32x2(pack_f32x2(rr[2 * q], rr[2 * q + 1]), f2);
                            const float2 fv = unpack_f32x2(v);
                            rr[2 * q] = __float_as_uint(fv.x);
                            rr[2 * q + 1] = __float_as_uint(fv.y);
                        }
                        tmem_st_32x32b_x32(ta + u * 32, rr);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(corr_done(x));
            }
        }
        // O = O_X svm / l, bf16
#pragma unroll
        for (int x = 0; x < 2; x++) {
            const int nx = x ? nB : nA;
            const int64_t row = q0 + x * AT_ROWS + r;
            const bool row_ok = row < p.seq_q;
            float scale = 0.0f;
            bool have = false;
            if (ok && nx > 0) {
                ok = __all_sync(0xFFFFFFFFu, at_wait(o_done(x), (nx - 1) & 1u)) &&
                     __all_sync(0xFFFFFFFFu, at_wait(l_full(x), 0));
                if (!ok) break;
                tc_fence_after();
                const float l = ld_shared_f32(sbase + A2_L_OFF + (x * 128 + r) * 4);
                scale = l > 0.0f ? svm / l : 0.0f;
                have = true;
            }
            if (!ok) break;
            uint16_t* o = reinterpret_cast<uint16_t*>(p.o) + row * p.ldo + static_cast<int64_t>(h) * AT_D;
#pragma unroll
            for (int u = 0; u < 4; u++) {
                uint32_t rr[32];
                if (have) {
                    tmem_ld_32x32b_x32(tmem + lane_off + 256 + x * 128 + u * 32, rr);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; i++) rr[i] = 0u;
                }
                if (row_ok) {
#pragma unroll
                    for (int c8 = 0; c8 < 4; c8++) {
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(rr[c8 * 8 + 2 * i]) * scale,
                                                                      __uint_as_float(rr[c8 * 8 + 2 * i + 1]) * scale);
                            w[i] = *reinterpret_cast<uint32_t*>(&h2);
                        }
                        *reinterpret_cast<uint4*>(o + u * 32 + c8 * 8) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t read_and_clear_attn_status(int* status) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(status, g_attn_status, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int));
}

#ifndef FP8BS_ATTN_V2
#define FP8BS_ATTN_V2 1
#endif

cudaError_t launch_fp8_attn_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const AttnParams& p, cudaStream_t st) {
    if (FP8BS_ATTN_V2) {
        auto k = k_fp8_attn_fwd2;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, A2_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        const int64_t qt = (p.seq_q + 2 * AT_ROWS - 1) / (2 * AT_ROWS);
        k<<<dim3(static_cast<unsigned>(qt), static_cast<unsigned>(p.hq)), A2_THREADS, A2_SMEM_BYTES, st>>>(
            tmQ, tmK, tmV, p);
        return cudaGetLastError();
    }
    auto k = k_fp8_attn_fwd;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t qt = (p.seq_q + AT_ROWS - 1) / AT_ROWS;
    k<<<dim3(static_cast<unsigned>(qt), static_cast<unsigned>(p.hq)), AT_THREADS, AT_SMEM_BYTES, st>>>(tmQ, tmK,
                                                                                                        tmV, p);
    return cudaGetLastError();
}

}  // namespace fp8bs
