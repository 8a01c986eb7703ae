// gemm.cu -- block-scaled FP8 GEMM on sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// Y = deq(A) . deq(B)^T with fp32 accumulation: the product of the FP8 linear
// layer ("NVIDIA NeMo RL logra una aceleracion del 48%...", hotbookzone.com,
// "El avance tecnico": 1x128 activation tiles and 128x128 weight tiles, E4M3,
// linear layers in FP8 math) for fprop, dgrad, wgrad and the grouped
// (mixture-of-experts) form.
//
// Kernel design (one persistent CTA per SM, 3 warpgroups = 12 warps):
//   warp 0      TMA producer: per 128-deep K block, one 128x128 A tile and
//               one 256x128 B tile (8-bit, 128-byte swizzle) into a 4-stage
//               shared-memory ring.
//   warp 1      TMEM owner and MMA issuer: per K block, 4 x
//               tcgen05.mma.kind::f8f6f4 (M=128, K=32) over the 256 columns,
//               as one N=256 slice (H = 1: a ring of two 256-column TMEM
//               buffers) or two N=128 slices (H = 2: four 128-column buffers).
//   warp 2      idle.
//   warp 3      scales: per K block, the products sA(row) * sB(column block)
//               for the tile's 128 rows into a shared-memory slot of the
//               block's TMEM buffer (loaded a few blocks ahead), its lanes
//               then joining that buffer's "full" barrier with the MMA
//               commit; with per-column B scales (1x128 B) it instead loads
//               the raw scale rows into a shared-memory ring.
//   warps 4..11 epilogue ("promotion"): each thread owns one output row (its
//               TMEM lane) and 128 columns; per K block it waits once for
//               the partial and its scale, loads the fp32 partial from TMEM
//               and folds it into fp32 registers: acc = fma(partial, sA * sB,
//               acc), two columns per packed f32x2 FMA.  At the end of a tile
//               it stores bf16 or fp32, or quantizes (optionally after
//               SwiGLU) to the next linear's FP8 operand.
// Register split (setmaxnreg): the block launches with 168 registers per
// thread (384 x 168 = 64512); the first warpgroup releases down to 104 and the
// two epilogue warpgroups grow to 200: 128 x 104 + 256 x 200 = 64512.
// A TMEM buffer goes back to the MMA right after the epilogue's last load of
// it, so the MMAs of the next block(s) overlap the promotion arithmetic.
// When both operands have one scale per tensor the whole K accumulates in
// TMEM and is scaled once ("promote every K").
// Operands may be stored K-major or MN-major (transposed storage, used by
// dgrad/wgrad); the instruction descriptor's major bits and the shared-memory
// descriptor strides select the layout.
//
// Every mbarrier wait is bounded (a few seconds of %globaltimer); a role
// that gives up records FP8BS_ERR_DEVICE_TIMEOUT in g_status, waits (bounded)
// for its own asynchronous work and leaves; TMEM is always freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fp8_math.cuh"
#include "gemm_kernels.h"
#include "ptx_sm100.cuh"

namespace fp8bs {

__device__ int g_status;  // 0 = ok, else a negative fp8bs status

namespace {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int STAGES = 4;
constexpr uint32_t A_STAGE = BM * BK;   // 16 KiB
constexpr uint32_t B_STAGE = BN * BK;   // 32 KiB
constexpr uint32_t STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int NUM_THREADS = 384;
constexpr int EPI_WARP0 = 4;
// setmaxnreg split of the 384 x 168 registers a CTA is launched with: the
// four control warps and the eight epilogue warps.  The control warps
// (producer, MMA, store / loader, scale warp) spill at 56 registers in most
// instances, which costs 5-10 %; the SwiGLU and per-column-B epilogues need
// the 224.
constexpr int REGS_LOW = 64, REGS_HIGH = 216;         // 128*64 + 256*216 <= 384*168
constexpr int REGS_LOW_WIDE = 56, REGS_HIGH_WIDE = 224;   // 128*56 + 256*224 == 384*168
static_assert(128 * REGS_LOW + 256 * REGS_HIGH <= 384 * 168, "register split");
static_assert(128 * REGS_LOW_WIDE + 256 * REGS_HIGH_WIDE <= 384 * 168, "register split");
constexpr int NUM_EPI_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;
#ifndef FP8BS_RASTER_M
#define FP8BS_RASTER_M 16
#endif
constexpr int RASTER_M = FP8BS_RASTER_M;   // m-slots per rasterization group
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;

// Each K block's MMAs run as H slices of N = 256 / H columns, each into its
// own TMEM buffer of a ring of 512 / (256 / H) buffers: H = 1 (two 256-column
// buffers) for the promotion epilogue, whose per-block work fits inside one
// MMA block; H = 2 (four 128-column buffers, each epilogue warpgroup
// following its own half) where the epilogue's per-block work is longer
// (per-column B scales), trading MMA rate (N = 128) for slack.
#ifndef FP8BS_HALVES
#define FP8BS_HALVES 1
#endif
#ifndef FP8BS_BCOL_HALVES
#define FP8BS_BCOL_HALVES 1
#endif
constexpr int HALVES = FP8BS_HALVES;
constexpr int BCOL_HALVES = FP8BS_BCOL_HALVES;
constexpr int MAX_TBUFS = 4;
// per-column B scales (1x128 B): a ring of BSF_SLOTS K blocks, each slot the
// tile's 256 B column scales (1 KiB) and, for a 1x128 A, its 128 row scales
constexpr int BSF_SLOTS = 4;
constexpr uint32_t BSF_SLOT_BYTES = 1536;
// promotion products (in the B-scale ring's space, unused by those kernels):
// per TMEM buffer a slot of the scale products of its 128 rows for two
// column parts (the two 128-column halves, or SwiGLU's gate and up blocks);
// then, with a 1x128 A scale table, a ring of SR_SLOTS slots, slot i %
// SR_SLOTS holding the A scales of K block i of this CTA for the tile's rows
// [r0, r0 + 132), r0 = its first row rounded down to a multiple of 4: the
// producer copies them (one bulk copy) along with the block's operand tiles
constexpr uint32_t SC_SLOT_BYTES = 2 * 128 * 4;
constexpr int SR_SLOTS = BSF_SLOTS;   // barriers: bsf_full = ready, bsf_empty = free
constexpr uint32_t SR_SLOT_BYTES = 132 * 4;
static_assert(2 * SC_SLOT_BYTES + SR_SLOTS * SR_SLOT_BYTES <= BSF_SLOTS * BSF_SLOT_BYTES,
              "scale slots fit the B-scale ring");
// output staging: 2 KiB sub-slabs (32 rows x 64 B, 64-B swizzle), one or four
// per epilogue warp
constexpr uint32_t OUT_SUB = 2048;
constexpr uint32_t OUT_SLAB = OUT_SUB;   // the MX kernel's slab
// amax exchange of the SwiGLU epilogue: [tile parity][column half][row] fp32
constexpr uint32_t XCHG_BYTES = 2 * 2 * 128 * 4;

// Shared memory of k_fp8_gemm: [align pad][A ring][B ring][barriers][tmem
// addr][group tables][output slabs][SwiGLU exchange][B-scale ring], for S
// operand stages and SUBS output sub-slabs per epilogue warp.  A K block
// waits for its operand tiles about four blocks' time (their copy latency),
// so four stages keep the MMA fed; with one sub-slab a tile's store passes
// wait in turn for the previous pass's store to read the slab.  Products
// with few K blocks per tile (at most SHORT_K_BLOCKS) store a tile every few
// blocks: their kernel keeps three stages and four sub-slabs, so a tile's
// four store passes never wait.
template <int S, int SUBS>
struct GemmLayout {
    static constexpr int kStages = S;
    static constexpr int kSubs = SUBS;
    static constexpr uint32_t kBarOff = S * STAGE_BYTES;
    // full, empty, tfull, tempty, done, xchg[4], bsf_full, bsf_empty,
    // st_full[8], st_free[8]
    static constexpr int kNumBars = 2 * S + 2 * MAX_TBUFS + 1 + 4 + 2 * BSF_SLOTS + 2 * NUM_EPI_WARPS;
    static constexpr uint32_t kTmemSlotOff = kBarOff + kNumBars * 8;
    static constexpr uint32_t kTableOff = (kTmemSlotOff + 16 + 15) & ~15u;
    static constexpr uint32_t kSlab = SUBS * OUT_SUB;
    static constexpr uint32_t kOutOff = (kTableOff + 2 * (kMaxGroups + 1) * 4 + 1023) & ~1023u;
    static constexpr uint32_t kXchgOff = kOutOff + NUM_EPI_WARPS * kSlab;
    static constexpr uint32_t kBsfOff = kXchgOff + XCHG_BYTES;
    static constexpr uint32_t kSmemBytes = 1024 + kBsfOff + BSF_SLOTS * BSF_SLOT_BYTES;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};
constexpr int SHORT_K_BLOCKS = 16;
template <bool SHORT_K>
using GemmLayoutFor = GemmLayout<SHORT_K ? STAGES - 1 : STAGES, SHORT_K ? 4 : 1>;

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t n = 0;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++n & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ bool wait_or_flag(uint32_t bar, uint32_t parity) {
    if (wait_bounded(bar, parity, WAIT_LIMIT_NS)) return true;
    atomicExch(&g_status, kStatusDeviceTimeout);
    return false;
}

struct Tile {
    int g, row0, row_end, nt;
};

// Tile t -> (group, first row, row limit, n-tile).  Tiles are rasterized in
// groups of RASTER_M m-slots: consecutive tiles walk the m-slots of a group
// first, then the n-tiles, so the CTAs in flight share A and B tiles in L2.
__device__ __forceinline__ Tile decode_tile(int t, int total_slots, int tiles_n, int G,
                                            const int* s_slot, const int* s_off) {
    const int per = RASTER_M * tiles_n;
    const int gm = t / per;
    const int r = t - gm * per;
    const int slot0 = gm * RASTER_M;
    const int gsz = min(RASTER_M, total_slots - slot0);
    const int nt = r / gsz;
    const int slot = slot0 + (r - nt * gsz);
    int lo = 0, hi = G;  // largest g with s_slot[g] <= slot
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_slot[mid] <= slot) lo = mid; else hi = mid;
    }
    Tile tl;
    tl.g = lo;
    tl.row0 = s_off[lo] + (slot - s_slot[lo]) * BM;
    tl.row_end = s_off[lo + 1];
    tl.nt = nt;
    return tl;
}

__device__ __forceinline__ float ld_scale(const float* p) { return __ldg(p); }
// a scale load kept in program order with the surrounding shared-memory
// accesses (bounds how many are in flight)
__device__ __forceinline__ float ld_scale_ordered(const float* p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}

// One warp's 32 rows x 128 columns of a finished tile as bf16 into its four
// 2 KiB sub-slabs (32 rows x 64 B each, 64-B swizzle: 16-B chunk c of row r
// at chunk c ^ (r/2)%4), the layout the output tensor map's TMA store reads.
__device__ __forceinline__ void stage_tile_bf16(const uint64_t (&acc)[64], uint32_t slab, int lane) {
    const uint32_t sw = (lane >> 1) & 3;
#pragma unroll
    for (int ps = 0; ps < 4; ps++) {
        const uint32_t rbase = slab + static_cast<uint32_t>(ps) * OUT_SUB + lane * 64;
#pragma unroll
        for (int c = 0; c < 4; c++) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const float2 f = unpack_f32x2(acc[ps * 16 + c * 4 + i]);
                __nv_bfloat162 h = __floats2bfloat162_rn(f.x, f.y);
                w[i] = *reinterpret_cast<uint32_t*>(&h);
            }
            st_shared_v4(rbase + ((c ^ sw) << 4), w[0], w[1], w[2], w[3]);
        }
    }
}

// Store one warp's 32 rows x 128 columns of a finished tile (acc = 128 fp32
// as packed pairs): TMA bulk stores of 32 x 64-byte boxes staged in the warp's
// `subs` 2 KiB sub-slabs when the warp's 32 rows all belong to the tile's
// group (TMA clips only at the tensor edge), otherwise masked direct stores.
__device__ __forceinline__ void store_tile(const GemmParams& p, const CUtensorMap& tmY,
                                           const uint64_t (&acc)[64], const Tile& tl, int64_t row,
                                           bool row_ok, int64_t col0, int quarter, int lane,
                                           uint32_t slab, int subs) {
    const int64_t wrow0 = static_cast<int64_t>(tl.row0) + quarter * 32;
    if (p.tma_store && (p.offsets == nullptr || wrow0 + 32 <= tl.row_end) && p.out_bf16 && subs == 4) {
        // bf16 with four sub-slabs: the whole 32 x 128 block at once -- the
        // four slabs written, one proxy fence, four stores issued together
        const uint32_t sw = (lane >> 1) & 3;          // 64-B swizzle: chunk ^= (row/2)%4
        if (lane == 0) bulk_wait_group_read0();       // this warp's earlier stores have read their slabs
        __syncwarp();
#pragma unroll
        for (int ps = 0; ps < 4; ps++) {
            const uint32_t rbase = slab + static_cast<uint32_t>(ps) * OUT_SUB + lane * 64;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const float2 f = unpack_f32x2(acc[ps * 16 + c * 4 + i]);
                    __nv_bfloat162 h = __floats2bfloat162_rn(f.x, f.y);
                    w[i] = *reinterpret_cast<uint32_t*>(&h);
                }
                st_shared_v4(rbase + ((c ^ sw) << 4), w[0], w[1], w[2], w[3]);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int ps = 0; ps < 4; ps++)
                tma_store_2d(&tmY, slab + static_cast<uint32_t>(ps) * OUT_SUB, static_cast<int32_t>(col0 + ps * 32),
                             static_cast<int32_t>(wrow0));
            bulk_commit_group();
        }
    } else if (p.tma_store && (p.offsets == nullptr || wrow0 + 32 <= tl.row_end)) {
        const uint32_t sw = (lane >> 1) & 3;          // 64-B swizzle: chunk ^= (row/2)%4
        const int passes = p.out_bf16 ? 4 : 8;        // 32 bf16 or 16 fp32 columns each
#pragma unroll
        for (int ps = 0; ps < 8; ps++) {
            if (ps >= passes) break;
            // pass ps uses sub-slab ps % subs, free once the store issued from
            // it subs passes ago has read it
            const uint32_t sub = slab + static_cast<uint32_t>(ps % subs) * OUT_SUB;
            const uint32_t rbase = sub + lane * 64;
            if (lane == 0) {
                if (subs == 4) bulk_wait_group_read3();
                else bulk_wait_group_read0();
            }
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t w[4];
                if (p.out_bf16) {
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const float2 f = unpack_f32x2(acc[ps * 16 + c * 4 + i]);
                        __nv_bfloat162 h = __floats2bfloat162_rn(f.x, f.y);
                        w[i] = *reinterpret_cast<uint32_t*>(&h);
                    }
                } else {
                    const float2 a = unpack_f32x2(acc[ps * 8 + c * 2]);
                    const float2 b = unpack_f32x2(acc[ps * 8 + c * 2 + 1]);
                    w[0] = __float_as_uint(a.x); w[1] = __float_as_uint(a.y);
                    w[2] = __float_as_uint(b.x); w[3] = __float_as_uint(b.y);
                }
                st_shared_v4(rbase + ((c ^ sw) << 4), w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&tmY, sub, static_cast<int32_t>(col0 + ps * (p.out_bf16 ? 32 : 16)),
                             static_cast<int32_t>(wrow0));
                bulk_commit_group();
            }
        }
    } else if (row_ok) {
        if (p.out_bf16) {
            uint16_t* y = reinterpret_cast<uint16_t*>(p.y) + row * p.ldy + col0;
#pragma unroll
            for (int j = 0; j < 128; j += 8) {
                if (col0 + j < p.N) {
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const float2 f = unpack_f32x2(acc[j / 2 + i]);
                        __nv_bfloat162 h = __floats2bfloat162_rn(f.x, f.y);
                        w[i] = *reinterpret_cast<uint32_t*>(&h);
                    }
                    *reinterpret_cast<uint4*>(y + j) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        } else {
            float* y = reinterpret_cast<float*>(p.y) + row * p.ldy + col0;
#pragma unroll
            for (int j = 0; j < 128; j += 4) {
                if (col0 + j < p.N) {
                    const float2 a = unpack_f32x2(acc[j / 2]), b = unpack_f32x2(acc[j / 2 + 1]);
                    *reinterpret_cast<float4*>(y + j) = make_float4(a.x, a.y, b.x, b.y);
                }
            }
        }
    }
}

// SwiGLU on one thread's 128 accumulator columns: columns 0-63 hold gate
// values and 64-127 the up values of the same 64 output columns; the
// results h = silu(gate) * up, silu(g) = g / (1 + e^-g), replace acc[0..31].
// The exponential and the division are the fast hardware forms (__expf,
// __fdividef: relative error about 5e-7 + 4e-8 |g|), since this runs on
// the critical path between tiles; the result is quantized to 8 bits.
// (g < -88: e^-g = inf and g / inf = -0.)
__device__ __forceinline__ void swiglu_inplace(uint64_t (&acc)[64]) {
#pragma unroll
    for (int i = 0; i < 32; i++) {
        const float2 g = unpack_f32x2(acc[i]);
        const float2 u = unpack_f32x2(acc[32 + i]);
        const float hx = __fdividef(g.x, 1.0f + __expf(-g.x)) * u.x;
        const float hy = __fdividef(g.y, 1.0f + __expf(-g.y)) * u.y;
        acc[i] = pack_f32x2(__float_as_uint(hx), __float_as_uint(hy));
    }
}

// Quantize one thread's first `nv` (128 or 64) output values of its row with
// the reciprocal block scale r and store the codes: TMA bulk stores of
// 32-row x 64-byte slabs as for the float output, else masked direct stores.
__device__ __forceinline__ void store_tile_q(const GemmParams& p, const CUtensorMap& tmY,
                                             const uint64_t (&acc)[64], int nv, float r,
                                             const Tile& tl, int64_t row, bool row_ok,
                                             int64_t qcol0, int quarter, int lane, uint32_t slab) {
    const int64_t wrow0 = static_cast<int64_t>(tl.row0) + quarter * 32;
    const int fmt = p.q_fmt;
    if (p.tma_store && (p.offsets == nullptr || wrow0 + 32 <= tl.row_end)) {
        const uint32_t rbase = slab + lane * 64;
        const uint32_t sw = (lane >> 1) & 3;          // 64-B swizzle: chunk ^= (row/2)%4
#pragma unroll
        for (int ps = 0; ps < 2; ps++) {
            if (ps * 64 >= nv) break;
            if (lane == 0) bulk_wait_group_read0();   // slab free again
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 4; c++) {            // 16 columns per 16-byte chunk
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const float2 a = unpack_f32x2(acc[ps * 32 + c * 8 + 2 * i]);
                    const float2 b = unpack_f32x2(acc[ps * 32 + c * 8 + 2 * i + 1]);
                    w[i] = quant4_rt(a.x, a.y, b.x, b.y, r, fmt);
                }
                st_shared_v4(rbase + ((c ^ sw) << 4), w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&tmY, slab, static_cast<int32_t>(qcol0 + ps * 64), static_cast<int32_t>(wrow0));
                bulk_commit_group();
            }
        }
    } else if (row_ok) {
        uint8_t* y = reinterpret_cast<uint8_t*>(p.y) + row * p.ldy + qcol0;
#pragma unroll
        for (int j = 0; j < 128; j += 16) {
            if (j >= nv) break;
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const float2 a = unpack_f32x2(acc[j / 2 + 2 * i]);
                const float2 b = unpack_f32x2(acc[j / 2 + 2 * i + 1]);
                w[i] = quant4_rt(a.x, a.y, b.x, b.y, r, fmt);
            }
            *reinterpret_cast<uint4*>(y + j) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// End of a tile in the epilogue: the float store, or (quantized output)
// optional SwiGLU, the block amax, the 1x128 scale and the codes.  With
// SwiGLU a 1x128 output block spans the two threads of a row (warps w and
// w + 4): each publishes its half's amax in shared memory and both wait,
// bounded, on their lane quarter's exchange barrier (64 arrivals per tile;
// two buffers by tile parity).  Returns false if that wait timed out.
template <bool SWIGLU>
__device__ __forceinline__ bool finish_tile(const GemmParams& p, const CUtensorMap& tmY,
                                            uint64_t (&acc)[64], const Tile& tl, int64_t row,
                                            bool row_ok, int64_t col0, int quarter, int half,
                                            int lane, uint32_t slab, uint32_t xbuf, uint32_t xbar,
                                            uint32_t tile_par, int subs = 1) {
    if (!p.out_q) {
        store_tile(p, tmY, acc, tl, row, row_ok, col0, quarter, lane, slab, subs);
        return true;
    }
    int nv = 128;
    int64_t qcol0 = col0, blk_col = col0;
    if (SWIGLU) {
        swiglu_inplace(acc);
        nv = 64;
        blk_col = static_cast<int64_t>(tl.nt) * 128;
        qcol0 = blk_col + half * 64;
    }
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 64; i++) {
        if (2 * i >= nv) break;
        const float2 f = unpack_f32x2(acc[i]);
        am = fmaxf(am, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
    if (SWIGLU) {
        const int lrow = quarter * 32 + lane;
        st_shared_f32(xbuf + ((tile_par * 2 + half) * 128 + lrow) * 4, am);
        mbar_arrive(xbar);
        if (!__all_sync(0xFFFFFFFFu, wait_or_flag(xbar, tile_par))) return false;
        am = fmaxf(am, ld_shared_f32(xbuf + ((tile_par * 2 + (half ^ 1)) * 128 + lrow) * 4));
    }
    if (blk_col < p.n_out) {
        const float s = block_scale_rt(am, p.q_fmt, p.q_mode);
        store_tile_q(p, tmY, acc, nv, __frcp_rn(s), tl, row, row_ok, qcol0, quarter, lane, slab);
        if (row_ok && (!SWIGLU || half == 0)) p.sq[(blk_col / 128) * p.a_rows + row] = s;
    }
    return true;
}

template <bool A_MN, bool B_MN, bool SWIGLU, bool B_COL, int H, bool SHORT_K = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_fp8_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmY, const GemmParams p) {
    constexpr int MMA_N = BN / H;
    constexpr int TBUFS = 512 / MMA_N;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sA = sbase;
    using L = GemmLayoutFor<SHORT_K>;
    constexpr int STAGES = L::kStages;
    constexpr bool WIDE_EPI = SWIGLU || B_COL;   // epilogues that need 224 registers
    constexpr int R_LOW = WIDE_EPI ? REGS_LOW_WIDE : REGS_LOW;
    constexpr int R_HIGH = WIDE_EPI ? REGS_HIGH_WIDE : REGS_HIGH;
    const uint32_t sB = sbase + STAGES * A_STAGE;
    const uint32_t bars = sbase + L::kBarOff;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bars + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bars + 8u * (2 * STAGES + MAX_TBUFS + b); };
    const uint32_t done_bar = bars + 8u * (2 * STAGES + 2 * MAX_TBUFS);
    auto xchg_bar = [&](int q) { return bars + 8u * (2 * STAGES + 2 * MAX_TBUFS + 1 + q); };
    auto bsf_full = [&](int q) { return bars + 8u * (2 * STAGES + 2 * MAX_TBUFS + 5 + q); };
    auto bsf_empty = [&](int q) { return bars + 8u * (2 * STAGES + 2 * MAX_TBUFS + 5 + BSF_SLOTS + q); };
    auto sr_ready = [&](int q) { return bsf_full(q); };   // (promotion products) a scale-ring
    auto sr_free = [&](int q) { return bsf_empty(q); };   // slot landed / was read
    // a bf16 block staged by epilogue warp w for the store warp / read out again
    auto st_full = [&](int w) { return bars + 8u * (2 * STAGES + 2 * MAX_TBUFS + 5 + 2 * BSF_SLOTS + w); };
    auto st_free = [&](int w) {
        return bars + 8u * (2 * STAGES + 2 * MAX_TBUFS + 5 + 2 * BSF_SLOTS + NUM_EPI_WARPS + w);
    };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlotOff);
    int* s_off = reinterpret_cast<int*>(smem + L::kTableOff);
    int* s_slot = s_off + (kMaxGroups + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.num_groups;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        for (int s = 0; s < STAGES; s++) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < TBUFS; b++) {
            // the MMA commit, plus the scale warp's 32 lanes (promotion products)
            mbar_init(tfull_bar(b), B_COL ? 1 : 33);
            mbar_init(tempty_bar(b), NUM_EPI_WARPS / H);   // the warps reading it
        }
        mbar_init(done_bar, 1);
        for (int q = 0; q < 4; q++) mbar_init(xchg_bar(q), 64);
        for (int q = 0; q < BSF_SLOTS; q++) {
            mbar_init(bsf_full(q), 1);   // the loader's (promotion: the producer's) expect_tx arrival
            // one arrival per epilogue warp (promotion: per scale-warp lane)
            mbar_init(bsf_empty(q), B_COL ? NUM_EPI_WARPS : 32);
        }
        for (int w = 0; w < NUM_EPI_WARPS; w++) {
            mbar_init(st_full(w), 1);
            mbar_init(st_free(w), 1);
        }
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    // group table: row offsets and the prefix count of 128-row m-slots
    // (row offsets are clamped into [0, a_rows], so no tile ever stores
    // outside Y whatever the device table holds)
    for (int i = threadIdx.x; i <= G; i += NUM_THREADS) {
        const int64_t o = p.offsets ? static_cast<int64_t>(p.offsets[i]) : (i == 0 ? 0 : p.M);
        s_off[i] = static_cast<int>(o < 0 ? 0 : (o > p.a_rows ? p.a_rows : o));
    }
    __syncthreads();
    if (warp == 2) {
        // prefix count of m-slots; a decreasing offset table (overlapping
        // groups, whose tiles would write the same rows) is rejected: every
        // CTA sees the same table, so all of them skip the product
        int carry = 0, bad = 0;
        if (lane == 0) s_slot[0] = 0;
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            int cnt = 0;
            if (g < G) {
                const int rows = s_off[g + 1] - s_off[g];
                bad |= rows < 0;
                cnt = (max(0, rows) + BM - 1) / BM;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xFFFFFFFFu, cnt, o);
                if (lane >= o) cnt += v;
            }
            if (g < G) s_slot[g + 1] = carry + cnt;
            carry += __shfl_sync(0xFFFFFFFFu, cnt, 31);
        }
        bad = __any_sync(0xFFFFFFFFu, bad);
        if (lane == 0) {
            tmem_slot[1] = bad;
            if (bad && blockIdx.x == 0) atomicCAS(&g_status, 0, kStatusBadOffsets);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total_slots = tmem_slot[1] ? 0 : s_slot[G];
    const int total_tiles = total_slots * p.tiles_n;
    const int nkb = static_cast<int>(p.K / BK);
    const int P = p.promote ? 1 : nkb;  // K blocks per TMEM partial
    // Products with few K blocks per tile (four output sub-slabs per warp)
    // and a plain bf16 output hand each finished block to warp 2, which
    // issues its TMA stores: issuing them takes ~1000 cycles behind the
    // operand copies in the TMA unit, time the epilogue warp now spends on
    // the next tile.
    const bool store_warp = !SWIGLU && !B_COL && L::kSubs == 4 && p.out_bf16 && !p.out_q && p.tma_store;

    if (warp < EPI_WARP0) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R_LOW));
      if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int issued = 0;
            for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
                const Tile tl = decode_tile(t, total_slots, p.tiles_n, G, s_slot, s_off);
                const int a_row = tl.row0;
                const int b_row = tl.g * p.b_rows_per_group + tl.nt * BN;
                // this tile's A scale rows for the scale ring
                const int64_t sr0 = tl.row0 & ~3;
                const uint32_t sr_bytes = static_cast<uint32_t>(
                    ((min(static_cast<int64_t>(tl.row0) + BM, p.a_rows) + 3) & ~3ll) - sr0) * 4u;
                for (int kb = 0; kb < nkb; kb++) {
                    if (!wait_or_flag(empty_bar(stage), phase ^ 1u)) { ok = false; break; }
                    if (!B_COL && p.sa_bulk) {
                        // the block's A scales, into the scale ring (their own barrier)
                        const int q = issued % SR_SLOTS;
                        if (!wait_or_flag(sr_free(q), ((static_cast<uint32_t>(issued) / SR_SLOTS) & 1u) ^ 1u)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(sr_ready(q), sr_bytes);
                        bulk_load_g2s(sbase + L::kBsfOff + TBUFS * SC_SLOT_BYTES + q * SR_SLOT_BYTES,
                                      p.sa + static_cast<int64_t>(kb) * p.a_rows + sr0, sr_bytes, sr_ready(q));
                    }
                    mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES);
                    const int kc = kb * BK;
                    const uint32_t dA = sA + stage * A_STAGE, dB = sB + stage * B_STAGE;
                    if (A_MN) tma_load_2d(dA, &tmA, a_row, kc, full_bar(stage));
                    else tma_load_2d(dA, &tmA, kc, a_row, full_bar(stage));
                    if (B_MN) {
                        tma_load_2d(dB, &tmB, b_row, kc, full_bar(stage));
                        tma_load_2d(dB + B_STAGE / 2, &tmB, b_row + 128, kc, full_bar(stage));
                    } else if (SWIGLU) {
                        // 64-row boxes: gate, up, gate + 64, up + 64 of this 128-column tile
                        const int gb = tl.g * p.b_rows_per_group + tl.nt * 128;
                        const int ub = gb + static_cast<int>(p.swiglu_i);
                        tma_load_2d(dB, &tmB, kc, gb, full_bar(stage));
                        tma_load_2d(dB + B_STAGE / 4, &tmB, kc, ub, full_bar(stage));
                        tma_load_2d(dB + B_STAGE / 2, &tmB, kc, gb + 64, full_bar(stage));
                        tma_load_2d(dB + 3 * (B_STAGE / 4), &tmB, kc, ub + 64, full_bar(stage));
                    } else {
                        tma_load_2d(dB, &tmB, kc, b_row, full_bar(stage));
                    }
                    issued++;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // drain: wait for the copies this thread issued on each stage
                for (int i = 0; i < STAGES && i < issued; i++) {
                    if (--stage < 0) { stage = STAGES - 1; phase ^= 1u; }
                    wait_bounded(full_bar(stage), phase, DRAIN_LIMIT_NS);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, group = 0;   // group = promotion group (P K blocks)
            bool ok = true, issued_mma = false;
            for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
                for (int kb = 0; kb < nkb; kb++) {
                    if (!wait_or_flag(full_bar(stage), phase)) { ok = false; break; }
                    const uint32_t aS = sA + stage * A_STAGE, bS = sB + stage * B_STAGE;
                    // two N=128 halves per K block, each into its own 128-column
                    // TMEM buffer of a 4-deep ring (chunk c = 2 * group + half)
#pragma unroll
                    for (int h = 0; h < H; h++) {
                        const uint32_t c = H * group + h, buf = c % TBUFS;
                        if (kb % P == 0) {
                            if (!wait_or_flag(tempty_bar(buf), ((c / TBUFS) & 1u) ^ 1u)) { ok = false; break; }
                        }
                        tc_fence_after();
                        const uint32_t d = tmem_base + buf * MMA_N;
#pragma unroll
                        for (int k4 = 0; k4 < BK / 32; k4++) {
                            // K-major: 32 K-bytes further inside the 128-byte swizzled
                            // row, 8-row groups 1024 B apart (SBO); half h starts 128
                            // rows (16 KiB) in.  MN-major: 32 K-rows further (4 swizzle
                            // atoms of 8 K-rows x 128 B, 1024 B apart), half h is the
                            // second TMA box; every MN-major descriptor spans a single
                            // 128-wide atom, so its MN-atom stride is never used and
                            // both offsets are 1024.
                            const uint64_t ad = A_MN ? smem_desc_sw128(aS + k4 * 4096, 1024, 1024)
                                                     : smem_desc_sw128(aS + k4 * 32, 16, 1024);
                            const uint32_t acc = (k4 > 0 || kb % P != 0) ? 1u : 0u;
                            if (B_MN) {   // one 128-wide TMA box per MMA (see above)
#pragma unroll
                                for (int q = 0; q < MMA_N / 128; q++)
                                    mma_f8f6f4(d + q * 128, ad,
                                               smem_desc_sw128(bS + (h * MMA_N / 128 + q) * (B_STAGE / 2) +
                                                                   k4 * 4096, 1024, 1024),
                                               p.idesc, acc);
                            } else {
                                mma_f8f6f4(d, ad, smem_desc_sw128(bS + h * (B_STAGE / 2) + k4 * 32, 16, 1024),
                                           p.idesc, acc);
                            }
                            issued_mma = true;
                        }
                        if (kb % P == P - 1) mma_commit(tfull_bar(buf));
                    }
                    if (!ok) break;
                    mma_commit(empty_bar(stage));
                    if (kb % P == P - 1) group++;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // after a timeout, let the MMAs already issued finish before TMEM
            // is released (on the normal path the epilogue consumed them all)
            if (!ok && issued_mma) {
                mma_commit(done_bar);
                wait_bounded(done_bar, 0, DRAIN_LIMIT_NS);
            }
        }
      } else if (B_COL && warp == 3) {
        // ------------- per-column B scale loader (1x128 B: table [K/128][N])
        // Per K block, two bulk copies into a ring slot: the tile's column
        // scales (row kb of B's table) and, for a 1x128 A, its row scales
        // (row kb of A's table); both tables are 16-byte aligned with row
        // pitches that are multiples of 16 bytes (checked on the host), and the
        // copies stop at the tables' ends.  A 128x128 or per-tensor A scale is
        // stored into the slot directly.  The epilogue warps free a slot once
        // they have read it.
        if (lane == 0) {
            int slot = 0;
            uint32_t ph = 0;
            bool ok = true;
            int issued = 0;
            for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
                const Tile tl = decode_tile(t, total_slots, p.tiles_n, G, s_slot, s_off);
                const int64_t n0 = static_cast<int64_t>(tl.nt) * BN;
                const uint32_t nb = static_cast<uint32_t>(min(static_cast<int64_t>(BN), p.N - n0)) * 4u;
                const uint32_t na = p.a_gran == 0
                    ? static_cast<uint32_t>(min(static_cast<int64_t>(BM), p.a_rows - tl.row0)) * 4u : 0u;
                for (int kb = 0; kb < nkb; kb++) {
                    if (!wait_or_flag(bsf_empty(slot), ph ^ 1u)) { ok = false; break; }
                    const uint32_t dst = sbase + L::kBsfOff + slot * BSF_SLOT_BYTES;
                    if (p.a_gran != 0)   // 128x128 / per-tensor A: its one scale of this K block
                        st_shared_f32(dst + 1024, ld_scale(p.sa + (p.a_gran == 1 ? (min(static_cast<int64_t>(tl.row0),
                                                                                        p.a_rows - 1) / 128) * nkb + kb : 0)));
                    mbar_arrive_expect_tx(bsf_full(slot), nb + na);
                    bulk_load_g2s(dst, p.sb + static_cast<int64_t>(kb) * p.N + n0, nb, bsf_full(slot));
                    if (na) bulk_load_g2s(dst + 1024, p.sa + static_cast<int64_t>(kb) * p.a_rows + tl.row0, na,
                                          bsf_full(slot));
                    issued++;
                    if (++slot == BSF_SLOTS) { slot = 0; ph ^= 1u; }
                }
            }
            if (!ok) {   // drain: let the copies already issued land
                for (int i = 0; i < BSF_SLOTS && i < issued; i++) {
                    if (--slot < 0) { slot = BSF_SLOTS - 1; ph ^= 1u; }
                    wait_bounded(bsf_full(slot), ph, DRAIN_LIMIT_NS);
                }
            }
        }
      } else if (warp == 2 && store_warp) {
        // ------------------------------------------------- tile store issuer
        // For every tile of this CTA and every epilogue warp whose 32 rows
        // lie inside the tile's group (the others store directly): wait for
        // the warp's staged block, issue its four TMA stores; once all of the
        // tile's stores have read their slabs, hand the slabs back.
        if (lane == 0) {
            uint32_t cnt[NUM_EPI_WARPS];
#pragma unroll
            for (int w = 0; w < NUM_EPI_WARPS; w++) cnt[w] = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
                const Tile tl = decode_tile(t, total_slots, p.tiles_n, G, s_slot, s_off);
                uint32_t used = 0;
#pragma unroll
                for (int w = 0; w < NUM_EPI_WARPS; w++) {
                    const int64_t wrow0 = static_cast<int64_t>(tl.row0) + (w & 3) * 32;
                    if (!ok || !(p.offsets == nullptr || wrow0 + 32 <= tl.row_end)) continue;
                    if (!wait_or_flag(st_full(w), cnt[w] & 1u)) { ok = false; continue; }
                    const uint32_t slab = sbase + L::kOutOff + w * L::kSlab;
                    const int64_t col0 = static_cast<int64_t>(tl.nt) * BN + (w >> 2) * 128;
#pragma unroll
                    for (int ps = 0; ps < 4; ps++)
                        tma_store_2d(&tmY, slab + static_cast<uint32_t>(ps) * OUT_SUB, static_cast<int32_t>(col0 + ps * 32),
                                     static_cast<int32_t>(wrow0));
                    bulk_commit_group();
                    used |= 1u << w;
                }
                if (used) {
                    bulk_wait_group_read0();   // the slabs have been read
#pragma unroll
                    for (int w = 0; w < NUM_EPI_WARPS; w++)
                        if (used & (1u << w)) {
                            mbar_arrive(st_free(w));
                            cnt[w]++;
                        }
                }
            }
            bulk_wait_group0();   // every store has landed
        }
      } else if (!B_COL && warp == 3) {
        // ------------------------------------- scale warp (promotion products)
        // Chunk c of this CTA (P K blocks of one tile, in the MMA's order)
        // goes to TMEM buffer c % TBUFS.  For its first K block the lanes
        // take the A scales of rows l + 32 e (lane l) -- from the scale ring
        // once its copy has landed, or else from global memory -- and the
        // two B scales; once the epilogue has released the
        // buffer (it read the slot's previous products before), they write
        // the products sA(row) * sB(part) into the buffer's slot and arrive
        // on its full barrier, so the epilogue waits once per chunk.
        static_assert(B_COL || H == 1, "one TMEM buffer per K block");
        const int cpt = nkb / P;
        const bool bulk = p.sa_bulk != 0;
        const uint32_t ring0 = sbase + L::kBsfOff + TBUFS * SC_SLOT_BYTES;
        uint32_t c = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
            const Tile tl = decode_tile(t, total_slots, p.tiles_n, G, s_slot, s_off);
            const int r0 = tl.row0 & ~3;
            uint32_t ro[4];   // rows l + 32 e (clamped) relative to r0
#pragma unroll
            for (int e = 0; e < 4; e++)
                ro[e] = static_cast<uint32_t>(min(static_cast<int64_t>(tl.row0) + lane + 32 * e, p.a_rows - 1) - r0);
            // the parts' weight row-blocks: columns 0-127 and 128-255 of the
            // tile, or SwiGLU's gate and up rows
            const int64_t n0 = static_cast<int64_t>(tl.nt) * BN;
            const int64_t nb0 = SWIGLU ? tl.nt : min(n0, p.N - 1) / 128;
            const int64_t nb1 = SWIGLU ? p.swiglu_i / 128 + tl.nt : min(n0 + 128, p.N - 1) / 128;
            const float* pb0 = p.sb;
            int64_t db = 0, sb_step = 0;   // part 1 at pb0 + db; per K block + sb_step
            if (p.b_gran == 1) {
                pb0 = B_MN ? p.sb + nb0 : p.sb + tl.g * p.b_scale_group_stride + nb0 * nkb;
                db = B_MN ? nb1 - nb0 : (nb1 - nb0) * nkb;
                sb_step = B_MN ? p.b_rblocks : 1;
            }
            for (int ci = 0; ci < cpt; ci++, c++) {
                const int64_t kb = static_cast<int64_t>(ci) * P;
                const float* pbk = pb0 + kb * sb_step;
                const float b0 = ld_scale(pbk), b1 = ld_scale(pbk + db);
                const uint32_t q = c % SR_SLOTS;
                const uint32_t ring = ring0 + q * SR_SLOT_BYTES;
                if (bulk) {
                    ok = __all_sync(0xFFFFFFFFu, wait_or_flag(sr_ready(q), (c / SR_SLOTS) & 1u));
                    if (!ok) break;
                } else {
                    // no ring copy: this lane stages its rows' A scales itself,
                    // row r's at sa + kb * ks + (r or its 128-row block) * rs,
                    // two loads in flight
                    const int64_t ks = p.a_gran == 0 ? p.a_rows : p.a_gran == 1 ? (A_MN ? p.a_rblocks : 1) : 0;
                    const int64_t rs = p.a_gran == 1 && !A_MN ? nkb : p.a_gran == 2 ? 0 : 1;
                    const int sh = p.a_gran == 1 ? 7 : 0;
                    const float* pak = p.sa + kb * ks;
                    const float v0 = ld_scale_ordered(pak + ((r0 + static_cast<int>(ro[0])) >> sh) * rs);
                    const float v1 = ld_scale_ordered(pak + ((r0 + static_cast<int>(ro[1])) >> sh) * rs);
                    st_shared_f32(ring + ro[0] * 4, v0);
                    st_shared_f32(ring + ro[1] * 4, v1);
                    const float v2 = ld_scale_ordered(pak + ((r0 + static_cast<int>(ro[2])) >> sh) * rs);
                    const float v3 = ld_scale_ordered(pak + ((r0 + static_cast<int>(ro[3])) >> sh) * rs);
                    st_shared_f32(ring + ro[2] * 4, v2);
                    st_shared_f32(ring + ro[3] * 4, v3);
                }
                float a[4];
#pragma unroll
                for (int e = 0; e < 4; e++) a[e] = ld_shared_f32(ring + ro[e] * 4);
                if (bulk) mbar_arrive(sr_free(q));   // each lane: its reads are done
                const uint32_t buf = c % TBUFS;
                ok = __all_sync(0xFFFFFFFFu, wait_or_flag(tempty_bar(buf), ((c / TBUFS) & 1u) ^ 1u));
                if (!ok) break;
                const uint32_t slot = sbase + L::kBsfOff + buf * SC_SLOT_BYTES;
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    st_shared_f32(slot + (lane + 32 * e) * 4, a[e] * b0);
                    st_shared_f32(slot + (128 + lane + 32 * e) * 4, a[e] * b1);
                }
                mbar_arrive(tfull_bar(buf));
            }
        }
      }
    } else if (B_COL) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R_HIGH));
        // ------------------------------ epilogue with per-column B scales
        // Every (row, column) needs its own product sa[row] * sb[col], so the
        // scales are read from shared memory each K block.  To keep that
        // traffic small each thread owns 4 rows x 32 columns (the 16x256b TMEM
        // load shape: rows 32 q + 16 lh + t/4 + 8 e, columns 8 c + 2 (t%4) + e'),
        // so it reads 32 B scales and 4 A scales per K block instead of 128.
        const int quarter = warp & 3;
        const int half = (warp - EPI_WARP0) >> 2;
        const int tq = lane >> 2, tc = lane & 3;
        uint32_t chunk = 0;
        int bslot = 0;
        uint32_t bph = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
            const Tile tl = decode_tile(t, total_slots, p.tiles_n, G, s_slot, s_off);
            const int64_t col0 = static_cast<int64_t>(tl.nt) * BN + half * 128;
            uint64_t acc[64];   // [row r (4)][column pair c (16)]
#pragma unroll
            for (int i = 0; i < 64; i++) acc[i] = 0;
            for (int kb = 0; kb < nkb; kb++) {
                const uint32_t buf = chunk % TBUFS;
                ok = __all_sync(0xFFFFFFFFu, wait_or_flag(tfull_bar(buf), (chunk / TBUFS) & 1u));
                if (!ok) break;
                ok = __all_sync(0xFFFFFFFFu, wait_or_flag(bsf_full(bslot), bph));
                if (!ok) break;
                tc_fence_after();
                const uint32_t slotb = sbase + L::kBsfOff + bslot * BSF_SLOT_BYTES;
                const uint32_t tb = tmem_base + buf * MMA_N + half * 128;
                float a[4];   // A scales of rows 16 lh + 8 e (+ t/4): a[2 lh + e]
#pragma unroll
                for (int r = 0; r < 4; r++)
                    a[r] = ld_shared_f32(slotb + 1024 +
                                         (p.a_gran == 0 ? (32 * quarter + 16 * (r >> 1) + 8 * (r & 1) + tq) * 4 : 0));
#pragma unroll
                for (int cp = 0; cp < 2; cp++) {
                    uint64_t sb2[8];   // B scale pairs of columns 64 cp + 8 k + 2 (t%4)
#pragma unroll
                    for (int k = 0; k < 8; k++) {
                        const uint2 b = ld_shared_v2(slotb + (half * 128 + 64 * cp + 8 * k + 2 * tc) * 4);
                        sb2[k] = pack_f32x2(b.x, b.y);
                    }
#pragma unroll
                    for (int lh = 0; lh < 2; lh++) {
                        const uint64_t s_lo = pack_f32x2(__float_as_uint(a[2 * lh]), __float_as_uint(a[2 * lh]));
                        const uint64_t s_hi =
                            pack_f32x2(__float_as_uint(a[2 * lh + 1]), __float_as_uint(a[2 * lh + 1]));
                        // 16 columns per TMEM round trip, each followed by its
                        // FMAs (measured faster than 8, 32 or 64 columns)
#pragma unroll
                        for (int hh = 0; hh < 4; hh++) {
                            uint32_t r[8];
                            tmem_ld_16x256b_x2(tb + (static_cast<uint32_t>(32 * quarter + 16 * lh) << 16) + 64 * cp + 16 * hh, r);
                            tmem_wait_ld();
                            if (lh == 1 && cp == 1 && hh == 3) {   // last load of this buffer: hand it back
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0) mbar_arrive(tempty_bar(buf));
                            }
#pragma unroll
                            for (int k = 0; k < 2; k++) {
                                const int kk = 2 * hh + k;
                                fma_f32x2(acc[(2 * lh) * 16 + 8 * cp + kk], pack_f32x2(r[4 * k], r[4 * k + 1]),
                                          mul_f32x2(sb2[kk], s_lo));
                                fma_f32x2(acc[(2 * lh + 1) * 16 + 8 * cp + kk], pack_f32x2(r[4 * k + 2], r[4 * k + 3]),
                                          mul_f32x2(sb2[kk], s_hi));
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bsf_empty(bslot));   // this warp read its scales
                if (++bslot == BSF_SLOTS) { bslot = 0; bph ^= 1u; }
                chunk++;
            }
            if (!ok) break;
            // direct stores, two columns at a time (8 B fp32 / 4 B bf16 per pair)
#pragma unroll
            for (int r = 0; r < 4; r++) {
                const int64_t row = static_cast<int64_t>(tl.row0) + 32 * quarter + 16 * (r >> 1) + tq + 8 * (r & 1);
                const bool rok = row < tl.row_end;
#pragma unroll
                for (int c = 0; c < 16; c++) {
                    const int64_t col = col0 + 8 * c + 2 * tc;
                    if (!rok || col >= p.N) continue;
                    const float2 v = unpack_f32x2(acc[r * 16 + c]);
                    if (p.out_bf16) {
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(v.x, v.y);
                        *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<uint16_t*>(p.y) + row * p.ldy + col) = h2;
                    } else {
                        *reinterpret_cast<float2*>(reinterpret_cast<float*>(p.y) + row * p.ldy + col) = v;
                    }
                }
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R_HIGH));
        // ----------------------------------------------------- epilogue
        const int quarter = warp & 3;           // TMEM lanes 32*quarter ..
        const int half = (warp - EPI_WARP0) >> 2;  // columns 128*half ..
        const int lrow = quarter * 32 + lane;
        const int cpt = nkb / P;                // TMEM chunks per tile
        // this thread's scale products in a slot: its half's part (SwiGLU:
        // the gate part for columns 0-63, the up part for 64-127)
        const uint32_t s_off0 = (SWIGLU ? 0u : static_cast<uint32_t>(half) * 512u) + lrow * 4;
        const uint32_t s_off1 = SWIGLU ? 512u + lrow * 4 : s_off0;
        uint32_t chunk = 0, tile_i = 0, ntma = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x, tile_i++) {
            const Tile tl = decode_tile(t, total_slots, p.tiles_n, G, s_slot, s_off);
            const int64_t row = static_cast<int64_t>(tl.row0) + lrow;
            const bool row_ok = row < tl.row_end;
            const int64_t col0 = static_cast<int64_t>(tl.nt) * BN + half * 128;

            uint64_t acc[64];   // 128 fp32 accumulators as packed pairs
#pragma unroll
            for (int i = 0; i < 64; i++) acc[i] = 0;
#pragma unroll 1
            for (int ci = 0; ci < cpt; ci++, chunk++) {
                const uint32_t buf = chunk % TBUFS;
                // one wait: the partial (MMA commit) and its scale products
                ok = __all_sync(0xFFFFFFFFu, wait_or_flag(tfull_bar(buf), (chunk / TBUFS) & 1u));
                if (!ok) break;
                tc_fence_after();
                const uint32_t slot = sbase + L::kBsfOff + buf * SC_SLOT_BYTES;
                const float s = ld_shared_f32(slot + s_off0);
                const float su = SWIGLU ? ld_shared_f32(slot + s_off1) : s;
                const uint64_t s2 = pack_f32x2(__float_as_uint(s), __float_as_uint(s));
                const uint64_t s2u = pack_f32x2(__float_as_uint(su), __float_as_uint(su));
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * MMA_N + half * 128;
                // 16 columns per TMEM round trip (measured faster than 8, 32
                // or 64: the loads and the FMAs interleave more finely); the
                // buffer is handed back right after the last load
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(taddr + j * 16, r);
                    tmem_wait_ld();
                    if (j == 7) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(tempty_bar(buf));
                    }
#pragma unroll
                    for (int q = 0; q < 8; q++)
                        fma_f32x2(acc[j * 8 + q], pack_f32x2(r[2 * q], r[2 * q + 1]), j < 4 ? s2 : s2u);
                }
            }
            if (!ok) break;
            const int64_t wrow0 = static_cast<int64_t>(tl.row0) + quarter * 32;
            if (store_warp && (p.offsets == nullptr || wrow0 + 32 <= tl.row_end)) {
                // stage the bf16 block for the store warp once it has read the
                // previous one out of this warp's slab
                const int w = warp - EPI_WARP0;
                if (ntma > 0) {
                    ok = __all_sync(0xFFFFFFFFu, wait_or_flag(st_free(w), (ntma - 1) & 1u));
                    if (!ok) break;
                }
                stage_tile_bf16(acc, sbase + L::kOutOff + w * L::kSlab, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(st_full(w));
                ntma++;
            } else {
                ok = finish_tile<SWIGLU>(p, tmY, acc, tl, row, row_ok, col0, quarter, half, lane,
                                 sbase + L::kOutOff + (warp - EPI_WARP0) * L::kSlab, sbase + L::kXchgOff,
                                 xchg_bar(quarter), tile_i & 1u, L::kSubs);
            }
        }
        if (lane == 0) bulk_wait_group0();   // every store of this warp has landed
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}


// ====================================================================== MX
// Power-of-two block scales applied by the tensor core: kind::mxf8f6f4 with
// UE8M0 scale factors in TMEM, so the whole K accumulates in TMEM with no
// promotion (the "block scaling accelerated by hardware" of Blackwell).
// Warp 0 loads each K block's operand tiles and (1x128 A scales) A's 128
// fp32 row scales by TMA; warp 2 waits for the stage to land and writes its
// UE8M0 words into the stage's scale area (B's two per-block scales come
// from a register ring), off the MMA's critical path; warp 1 copies them
// into a 4-slot TMEM ring with tcgen05.cp (ordered with its MMAs) and issues
// the block-scaled MMAs.  A's
// scale of row m sits at TMEM (lane m, column m/32) of its slot (the 128x128b
// copy fills all four columns of each lane); B's scale of column n sits at
// (lane 32*quarter + n%32, column 4 + n/32), one copy per lane quarter (the
// 32x128b.warpx4 copy).  One 256-column accumulator; the epilogue loads it,
// releases it and stores.
// per stage: A's raw fp32 scales (512 B, by TMA) at 0, SFA words 128x16 B at
// 512, SFB words 2 x 32x16 B at 2560 and 3072
constexpr uint32_t MX_SF_STAGE = 3584;
constexpr uint32_t MX_SF_OFF = STAGES * STAGE_BYTES;
constexpr uint32_t MX_BAR_OFF = MX_SF_OFF + STAGES * MX_SF_STAGE;
constexpr int MX_NUM_BARS = 3 * STAGES + 2 + 1 + 4;    // full, empty, sfready, tfull, tempty, done, xchg[4]
constexpr uint32_t MX_TMEMSLOT_OFF = MX_BAR_OFF + MX_NUM_BARS * 8;
constexpr uint32_t MX_TABLE_OFF = (MX_TMEMSLOT_OFF + 16 + 15) & ~15u;
constexpr uint32_t MX_OUT_OFF = (MX_TABLE_OFF + 16 + 1023) & ~1023u;
constexpr uint32_t MX_XCHG_OFF = MX_OUT_OFF + NUM_EPI_WARPS * OUT_SLAB;
constexpr uint32_t MX_SMEM_BYTES = 1024 + MX_XCHG_OFF + XCHG_BYTES;
static_assert(MX_SMEM_BYTES <= 232448, "shared memory budget (MX)");
constexpr uint32_t MX_SF_TMEM = 256;                   // scale-factor ring after the accumulator
constexpr int MX_SF_SLOTS = 4;                         // 16 columns each: SFA 4 + SFB 8
#ifndef FP8BS_MPF
#define FP8BS_MPF 8
#endif
constexpr int MPF = FP8BS_MPF;                         // producer scale prefetch (K blocks)
constexpr int MX_REGS_LOW = 96, MX_REGS_HIGH = 200;   // 128*96 + 256*200 <= 384*168 (88 / 208 spilled)

// UE8M0 code of a power-of-two fp32 scale (its exponent field), in all 4 bytes
__device__ __forceinline__ uint32_t ue8m0_word(float s) {
    return ((__float_as_uint(s) >> 23) & 0xFFu) * 0x01010101u;
}

template <bool SWIGLU, bool MX32>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_fp8_gemm_mx(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmSA,
                  const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sA = sbase, sB = sbase + STAGES * A_STAGE, sSF = sbase + MX_SF_OFF;
    const uint32_t bars = sbase + MX_BAR_OFF;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto sfready_bar = [&](int s) { return bars + 8u * (2 * STAGES + s); };
    const uint32_t tfull_bar = bars + 8u * (3 * STAGES);
    const uint32_t tempty_bar = bars + 8u * (3 * STAGES + 1);
    const uint32_t done_bar = bars + 8u * (3 * STAGES + 2);
    auto xchg_bar = [&](int q) { return bars + 8u * (3 * STAGES + 3 + q); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + MX_TMEMSLOT_OFF);
    int* s_off = reinterpret_cast<int*>(smem + MX_TABLE_OFF);
    int* s_slot = s_off + 2;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        for (int s = 0; s < STAGES; s++) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            mbar_init(sfready_bar(s), 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(tempty_bar, NUM_EPI_WARPS);
        mbar_init(done_bar, 1);
        for (int q = 0; q < 4; q++) mbar_init(xchg_bar(q), 64);
        fence_mbar_init();
        fence_proxy_async_smem();
        s_off[0] = 0;
        s_off[1] = static_cast<int>(p.M);
        s_slot[0] = 0;
        s_slot[1] = static_cast<int>((p.M + BM - 1) / BM);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total_slots = s_slot[1];
    const int total_tiles = total_slots * p.tiles_n;
    const int nkb = static_cast<int>(p.K / BK);
    const int64_t nkb64 = nkb;
    const int64_t nrbB = (p.N + 127) / 128;

    // A's 1x128 fp32 scales, or (MXFP8) A's E8M0 words, arrive by TMA
    const bool sa_tma = MX32 || p.a_gran == 0;

    if (warp < EPI_WARP0) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(MX_REGS_LOW));
      if (warp == 0) {
        // -------------------------------- producer: operand tiles + A's scale vector
        if (lane == 0) {
            if (sa_tma) tma_prefetch_desc(&tmSA);
            const uint32_t bytes = STAGE_BYTES + (sa_tma ? 512u : 0u);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int issued = 0;
            for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
                const Tile tl = decode_tile(t, total_slots, p.tiles_n, 1, s_slot, s_off);
                for (int kb = 0; kb < nkb; kb++) {
                    if (!wait_or_flag(empty_bar(stage), phase ^ 1u)) { ok = false; break; }
                    mbar_arrive_expect_tx(full_bar(stage), bytes);
                    tma_load_2d(sA + stage * A_STAGE, &tmA, kb * BK, tl.row0, full_bar(stage));
                    const uint32_t dB = sB + stage * B_STAGE;
                    if (SWIGLU) {   // 64-row boxes: gate, up, gate + 64, up + 64
                        const int gb = tl.nt * 128, ub = gb + static_cast<int>(p.swiglu_i);
                        tma_load_2d(dB, &tmB, kb * BK, gb, full_bar(stage));
                        tma_load_2d(dB + B_STAGE / 4, &tmB, kb * BK, ub, full_bar(stage));
                        tma_load_2d(dB + B_STAGE / 2, &tmB, kb * BK, gb + 64, full_bar(stage));
                        tma_load_2d(dB + 3 * (B_STAGE / 4), &tmB, kb * BK, ub + 64, full_bar(stage));
                    } else {
                        tma_load_2d(dB, &tmB, kb * BK, tl.nt * BN, full_bar(stage));
                    }
                    if (sa_tma)   // 128 fp32 row scales of this K block (rows contiguous)
                        tma_load_2d(sSF + stage * MX_SF_STAGE, &tmSA, tl.row0, kb, full_bar(stage));
                    issued++;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                for (int i = 0; i < STAGES && i < issued; i++) {
                    if (--stage < 0) { stage = STAGES - 1; phase ^= 1u; }
                    wait_bounded(full_bar(stage), phase, DRAIN_LIMIT_NS);
                }
            }
        }
      } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, tile_i = 0, kbg = 0;
            bool ok = true, issued_mma = false;
            for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x, tile_i++) {
                if (!wait_or_flag(tempty_bar, (tile_i & 1u) ^ 1u)) { ok = false; break; }
                for (int kb = 0; kb < nkb; kb++, kbg++) {
                    // scale words written (the converter saw the stage's TMA land)
                    if (!wait_or_flag(sfready_bar(stage), phase)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sf = sSF + stage * MX_SF_STAGE;
                    const uint32_t tsfa = tmem_base + MX_SF_TMEM + (kbg % MX_SF_SLOTS) * 16;
                    const uint32_t tsfb = tsfa + 4;
                    tmem_cp_128x128b(tsfa, smem_desc_rows16(sf + 512));
                    tmem_cp_32x128b_warpx4(tsfb, smem_desc_rows16(sf + 2560));
                    tmem_cp_32x128b_warpx4(tsfb + 4, smem_desc_rows16(sf + 3072));
                    const uint32_t aS = sA + stage * A_STAGE, bS = sB + stage * B_STAGE;
                    // MXFP8: each K = 32 slice reads its own scale byte of the
                    // words (A and B scale-factor ids = k4); otherwise the four
                    // bytes are equal and id 0 serves every slice
#pragma unroll
                    for (int k4 = 0; k4 < BK / 32; k4++)
                        mma_mxf8f6f4(tmem_base, smem_desc_sw128(aS + k4 * 32, 16, 1024),
                                     smem_desc_sw128(bS + k4 * 32, 16, 1024),
                                     MX32 ? (p.idesc | (static_cast<uint32_t>(k4) << 29) |
                                             (static_cast<uint32_t>(k4) << 4))
                                          : p.idesc,
                                     tsfa, tsfb, (kb > 0 || k4 > 0) ? 1u : 0u);
                    issued_mma = true;
                    mma_commit(empty_bar(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(tfull_bar);
            }
            if (!ok && issued_mma) {
                mma_commit(done_bar);
                wait_bounded(done_bar, 0, DRAIN_LIMIT_NS);
            }
        }
      } else if (MX32 && warp == 2) {
        // ------ MXFP8 scale staging: A's words (by TMA) and B's words (from a
        // register ring, 4 K blocks ahead) into the tcgen05.cp layouts
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        const uint32_t* sbw = reinterpret_cast<const uint32_t*>(p.sb);   // [K/128][N] words
        for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
            const Tile tl = decode_tile(t, total_slots, p.tiles_n, 1, s_slot, s_off);
            const int64_t n0 = static_cast<int64_t>(tl.nt) * BN;
            uint32_t bw[4][8];
            auto load_bw = [&](int kbi, uint32_t (&d)[8]) {
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    const int64_t n = n0 + 32 * c + lane;
                    d[c] = (kbi < nkb && n < p.N) ? __ldg(sbw + static_cast<int64_t>(kbi) * p.N + n) : 0u;
                }
            };
#pragma unroll
            for (int i = 0; i < 4; i++) load_bw(i, bw[i]);
            for (int kb0 = 0; ok && kb0 < nkb; kb0 += 4) {
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int kb = kb0 + i;
                    if (kb >= nkb) break;
                    ok = __all_sync(0xFFFFFFFFu, wait_or_flag(full_bar(stage), phase));
                    if (!ok) break;
                    const uint32_t sf = sSF + stage * MX_SF_STAGE;
#pragma unroll
                    for (int r = 0; r < 4; r++) {
                        const uint32_t w = __float_as_uint(ld_shared_f32(sf + (32 * r + lane) * 4));
                        st_shared_v4(sf + 512 + (32 * r + lane) * 16, w, w, w, w);
                    }
                    // word c of row `lane` feeds column 32 c + lane (+128 for the second copy)
                    st_shared_v4(sf + 2560 + lane * 16, bw[i][0], bw[i][1], bw[i][2], bw[i][3]);
                    st_shared_v4(sf + 3072 + lane * 16, bw[i][4], bw[i][5], bw[i][6], bw[i][7]);
                    load_bw(kb + 4, bw[i]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sfready_bar(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
        }
      } else if (!MX32 && warp == 2) {
        // ---------------- scale converter: UE8M0 words of each landed stage
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
            const Tile tl = decode_tile(t, total_slots, p.tiles_n, 1, s_slot, s_off);
            // weight row-blocks: columns 0-127 / 128-255 of the tile; with
            // SwiGLU the gate (nb0) and up (nb1) blocks of 64-column runs
            const int64_t nb0 = SWIGLU ? tl.nt : min(static_cast<int64_t>(2 * tl.nt), nrbB - 1);
            const int64_t nb1 = SWIGLU ? p.swiglu_i / 128 + tl.nt
                                         : min(static_cast<int64_t>(2 * tl.nt + 1), nrbB - 1);
            const int64_t arow = min(static_cast<int64_t>(tl.row0), p.a_rows - 1);
            // lane-uniform scale values of K block kb in register slot kb % MPF
            float ru[MPF], rb0[MPF], rb1[MPF];
            auto load_sf = [&](int kb, float& u, float& b0, float& b1) {
                u = p.a_gran == 1 ? ld_scale(p.sa + (arow / 128) * nkb64 + kb)
                                  : (p.a_gran == 2 ? ld_scale(p.sa) : 0.0f);
                b0 = p.b_gran == 1 ? ld_scale(p.sb + nb0 * nkb64 + kb) : ld_scale(p.sb);
                b1 = p.b_gran == 1 ? ld_scale(p.sb + nb1 * nkb64 + kb) : ld_scale(p.sb);
            };
#pragma unroll
            for (int i = 0; i < MPF; i++) load_sf(min(i, nkb - 1), ru[i], rb0[i], rb1[i]);
            for (int kb0 = 0; ok && kb0 < nkb; kb0 += MPF) {
#pragma unroll
                for (int i = 0; i < MPF; i++) {
                    const int kb = kb0 + i;
                    if (kb >= nkb) break;
                    ok = __all_sync(0xFFFFFFFFu, wait_or_flag(full_bar(stage), phase));
                    if (!ok) break;
                    const uint32_t sf = sSF + stage * MX_SF_STAGE;
#pragma unroll
                    for (int r = 0; r < 4; r++) {
                        const float v = sa_tma ? ld_shared_f32(sf + (32 * r + lane) * 4) : ru[i];
                        const uint32_t w = ue8m0_word(v);
                        st_shared_v4(sf + 512 + (32 * r + lane) * 16, w, w, w, w);
                    }
                    // word c of row `lane` feeds column 32 c + lane (+128 for the second copy)
                    const uint32_t w0 = ue8m0_word(rb0[i]), w1 = ue8m0_word(rb1[i]);
                    if (SWIGLU) {
                        st_shared_v4(sf + 2560 + lane * 16, w0, w0, w1, w1);
                        st_shared_v4(sf + 3072 + lane * 16, w0, w0, w1, w1);
                    } else {
                        st_shared_v4(sf + 2560 + lane * 16, w0, w0, w0, w0);
                        st_shared_v4(sf + 3072 + lane * 16, w1, w1, w1, w1);
                    }
                    if (kb + MPF < nkb) load_sf(kb + MPF, ru[i], rb0[i], rb1[i]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sfready_bar(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
        }
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(MX_REGS_HIGH));
        // ----------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int half = (warp - EPI_WARP0) >> 2;
        uint32_t tile_i = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x, tile_i++) {
            const Tile tl = decode_tile(t, total_slots, p.tiles_n, 1, s_slot, s_off);
            const int64_t row = static_cast<int64_t>(tl.row0) + quarter * 32 + lane;
            const bool row_ok = row < tl.row_end;
            const int64_t col0 = static_cast<int64_t>(tl.nt) * BN + half * 128;
            ok = __all_sync(0xFFFFFFFFu, wait_or_flag(tfull_bar, tile_i & 1u));
            if (!ok) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + half * 128;
            uint64_t acc[64];
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                uint32_t r[2][32];
                tmem_ld_32x32b_x32(taddr + j * 32, r[0]);
                tmem_ld_32x32b_x32(taddr + (j + 1) * 32, r[1]);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 2; u++)
#pragma unroll
                    for (int i = 0; i < 16; i++) acc[(j + u) * 16 + i] = pack_f32x2(r[u][2 * i], r[u][2 * i + 1]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar);       // accumulator free for the next tile
            ok = finish_tile<SWIGLU>(p, tmY, acc, tl, row, row_ok, col0, quarter, half, lane,
                             sbase + MX_OUT_OFF + (warp - EPI_WARP0) * OUT_SLAB, sbase + MX_XCHG_OFF,
                             xchg_bar(quarter), tile_i & 1u);
        }
        if (lane == 0) bulk_wait_group0();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// arrives at, with a limit of `limit_ns`; on expiry it records the timeout in
// g_status exactly as the GEMM roles do, and the kernel returns normally.
__global__ void k_wait_selftest(uint64_t limit_ns, int* out) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        const uint32_t b = smem_u32(&bar);
        mbar_init(b, 1);
        fence_mbar_init();
        const bool ok = wait_bounded(b, 0, limit_ns);
        if (!ok) atomicExch(&g_status, kStatusDeviceTimeout);
        *out = ok ? 1 : 0;
    }
}

__global__ void k_fill_f32(float* p, int64_t n, float v) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        p[i] = v;
}

}  // namespace

cudaError_t launch_fill_f32(float* p, int64_t n, float v, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    const int64_t blocks = (n + 255) / 256;
    k_fill_f32<<<static_cast<unsigned>(blocks < 1024 ? blocks : 1024), 256, 0, st>>>(p, n, v);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, int* out, cudaStream_t st) {
    k_wait_selftest<<<1, 32, 0, st>>>(limit_ns, out);
    return cudaGetLastError();
}


// kind::f8f6f4 instruction descriptor: D fp32 (bits 4-5 = 1), A/B formats
// (bits 7-9, 10-12: E4M3 = 0, E5M2 = 1), A/B major (bits 15, 16: 1 = MN),
// N >> 3 (bits 17-22), M >> 4 (bits 24-28).
uint32_t make_idesc_f8f6f4(int a_fmt, int b_fmt, bool a_mn, bool b_mn, int n) {
    uint32_t d = 0;
    d |= 1u << 4;
    d |= static_cast<uint32_t>(a_fmt & 7) << 7;
    d |= static_cast<uint32_t>(b_fmt & 7) << 10;
    d |= (a_mn ? 1u : 0u) << 15;
    d |= (b_mn ? 1u : 0u) << 16;
    d |= static_cast<uint32_t>(n >> 3) << 17;
    d |= static_cast<uint32_t>(BM >> 4) << 24;
    return d;
}

// kind::mxf8f6f4 (block-scaled) instruction descriptor: B / A scale-factor
// byte ids at bits 4-5 / 29-30 (0: the four bytes of a scale word are equal
// here), A/B formats at 7-9 / 10-12, N >> 3 at 17-22, scale type UE8M0 at
// bit 23, M >> 4 at 24-28; the accumulator is always fp32.
uint32_t make_idesc_mx(int a_fmt, int b_fmt, int n) {
    uint32_t d = 0;
    d |= static_cast<uint32_t>(a_fmt & 7) << 7;
    d |= static_cast<uint32_t>(b_fmt & 7) << 10;
    d |= static_cast<uint32_t>(n >> 3) << 17;
    d |= 1u << 23;
    d |= static_cast<uint32_t>(BM >> 4) << 24;
    return d;
}

cudaError_t launch_fp8_gemm_mx(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmY,
                               const CUtensorMap& tmSA, const GemmParams& p, int grid, cudaStream_t st) {
    auto k = p.mx32 ? k_fp8_gemm_mx<false, true> : p.swiglu ? k_fp8_gemm_mx<true, false> : k_fp8_gemm_mx<false, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MX_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    k<<<grid, NUM_THREADS, MX_SMEM_BYTES, st>>>(tmA, tmB, tmY, tmSA, p);
    return cudaGetLastError();
}

int gemm_tile_n() { return BN; }
int gemm_mma_n(bool b_col) { return BN / (b_col ? BCOL_HALVES : HALVES); }
int gemm_tile_m() { return BM; }

cudaError_t launch_fp8_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmY,
                            const GemmParams& p, bool a_mn, bool b_mn, int grid, cudaStream_t st) {
    // SwiGLU and per-column B scales run only on K-major operands (the host
    // checks it); the latter with BCOL_HALVES MMA slices per K block
    constexpr int h1 = HALVES, hb = BCOL_HALVES;
    // (the plain K-major product with few K blocks per tile: three stages,
    // four output sub-slabs)
    const bool short_k = !p.swiglu && p.b_gran != 0 && !a_mn && !b_mn && p.K / BK <= SHORT_K_BLOCKS;
    auto k = p.swiglu ? k_fp8_gemm<false, false, true, false, h1>
             : p.b_gran == 0 ? k_fp8_gemm<false, false, false, true, hb>
             : a_mn ? (b_mn ? k_fp8_gemm<true, true, false, false, h1> : k_fp8_gemm<true, false, false, false, h1>)
             : b_mn ? k_fp8_gemm<false, true, false, false, h1>
             : short_k ? k_fp8_gemm<false, false, false, false, h1, true> : k_fp8_gemm<false, false, false, false, h1>;
    const uint32_t smem = short_k ? GemmLayoutFor<true>::kSmemBytes : GemmLayoutFor<false>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k<<<grid, NUM_THREADS, smem, st>>>(tmA, tmB, tmY, p);
    return cudaGetLastError();
}

cudaError_t read_and_clear_status(int* status) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(status, g_status, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
}

}  // namespace fp8bs
