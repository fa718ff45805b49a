// Prefill path of the expert FFN: tcgen05 block-scaled grouped GEMM over the
// per-expert token groups, fed by TMA, accumulating in tensor memory.
//
// Source: tinyserve README, "How it works" item 6 -- batched prefill groups
// tokens by expert and loads each unique expert once; item 2 -- the expert
// runs directly on its quantised bytes (gate, up, down).  llama.cpp
// discussion "fixed GPU expert working set with Native CPU miss execution",
// prefill update -- grouped matrix products over a per-layer unique-expert
// pack.  Formats: OCP MX v1.0 (E4M3 activations and E2M1 weights, E8M0
// scale per 32 along K).
//
// Per layer call:
//   1. quant: x (bf16) -> MXFP8, rows gathered in grouped (perm) order;
//   2. gate/up GEMM: per expert e, rows [offsets[e], offsets[e+1]) of the
//      grouped activations times the expert's interleaved gate/up matrix;
//      epilogue h = bf16(silu(g) * u) -> MXFP8 (scale per 32 along I);
//   3. down GEMM: grouped h times the expert's down matrix; its epilogue is
//      the combine: out[token(row)] += w(row) * y(row) with float4 fp32
//      atomics, so the k terms of a token land in completion order (out is
//      zeroed first unless the caller accumulates into a residual stream).
// The GEMM launches use programmatic stream serialisation (each waits for
// its predecessor with griddepcontrol before touching global memory), and
// the pipeline roles wait on their mbarriers with the hardware-suspending
// try_wait, resuming the moment a phase completes.
//
// GEMM kernel (persistent, one CTA per SM, 16 warps in four warpgroups):
//   warp 0     TMA producer: 128x128-byte A tile (E4M3) and 256x128-element
//              B tile (E2M1, unpacked by TMA into the 16-byte-aligned layout
//              the f8f6f4 MMA reads) per stage, 128-byte swizzle;
//   warp 1     MMA issuer: tcgen05.mma kind::mxf8f6f4 block_scale 1X,
//              M=128 N=256 K=32, four per stage, into a tensor-memory
//              accumulator;
//   warps 4-7  scale-factor feeders: per group of eight stages, the E8M0
//              bytes of the tile's 128 activation rows and 256 weight rows
//              go into one of two tensor-memory slots, freed by an MMA
//              commit once the group that used the slot two groups back
//              has finished;
//   warps 8-15 epilogue: copy the finished accumulator into registers
//              (a half row per thread), hand it back to the MMA for the
//              next tile, and finish the tile from registers.
// Each stage costs the MMA a roughly fixed overhead for fetching fresh
// scale factors, so the widest tile the hardware takes (N = 256) gives the
// most products per stage; its accumulator then fills half of tensor
// memory, and the quick register copy stands in for a second accumulator.
// Tiles (expert, 128-row block, 256-column block) are enumerated on the
// device from the offsets; columns vary fastest so the CTAs working at the
// same time share an expert's activation rows and weight rows through L2
// (for a down launch whose output exceeds half of L2, within groups of a
// few column blocks, so that the output rows its combine adds into stay
// in L2 while they are being hit).
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstddef>
#include <mutex>

#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;           // rows (tokens) per tile
constexpr int kBN = 256;           // weight rows per tile
constexpr int kBK = 128;           // K elements per pipeline stage
constexpr int kStages = 4;
constexpr int kThreads = 512;      // four warpgroups
constexpr uint32_t kStageBytesA = kBM * kBK;   // E4M3: one byte per element
constexpr uint32_t kStageBytesB = kBN * kBK;   // E2M1 unpacked: 16 bytes per 16 elements in smem
constexpr uint32_t kTxBytesB = kBN * kBK / 2;  // ...of which TMA writes the 8 packed bytes per 16
constexpr uint32_t kTmemCols = 512;
// Tensor-memory columns: the fp32 accumulator at [0, kBN); then two
// scale-factor slots of 128 columns, each holding the factors of a group of
// eight K stages (the feeders write a whole group at once, which the MMA
// waits for once per group: fresh factors before every stage cost the
// tensor pipe about 200 cycles a stage), 16 columns per stage: A at +0 (4
// columns), B at +8 (kBN / 32 columns).  Row m of an operand keeps its
// stage's four E8M0 bytes in lane m % 32 of every lane quarter, column
// base + m / 32 (each quarter of the tensor core reads its own copy); byte
// j of that word belongs to the stage's j-th block of 32 and is picked by
// the MMA's scale-factor id.
constexpr uint32_t kColSf = kBN;
constexpr int kSfGroup = 8;   // K stages per scale-factor group
__host__ __device__ constexpr uint32_t sf_col_g(int gs, int s) { return kColSf + 16 * kSfGroup * gs + 16 * s; }
constexpr int kMaxExperts = MOE_MAX_EXPERTS;
constexpr int kYPad = 20;          // padded row of the epilogue's y staging tile (words)
static_assert(kBN % 64 == 0 && kBN / 32 <= 8, "tile width: whole chunk pairs, B scales in 8 columns");
static_assert(sf_col_g(2, 0) <= kTmemCols, "tensor-memory columns");
// Register split between the warpgroups (setmaxnreg): launched with
// kLaunchRegs per thread, warpgroup 0 (TMA, MMA) gives registers up to the
// scale-factor feeders (warpgroup 1) and the epilogue (warpgroups 2, 3),
// which holds a thread's half row of the accumulator in registers.
constexpr int kLaunchRegs = 65536 / kThreads;
constexpr int kRegsCtl = 48, kRegsSf = 144, kRegsEpi = 160;
static_assert(kRegsCtl + kRegsSf + 2 * kRegsEpi == 4 * kLaunchRegs, "register split sums to the launch's share");

constexpr int kMaxSlotTab = MOE_MAX_EXPERTS;  // experts of one launch when slots come by value

struct GemmParams {
    const int32_t* offsets;     // [E+1] grouped row ranges
    const int32_t* slot_of;     // [E] device slot map, or nullptr: slot_tab
    int32_t slot_tab[kMaxSlotTab];  // slot of each of the E experts (E <= kMaxSlotTab)
    int E, A, S;
    int K, KB;                  // reduction length and its 32-blocks
    int N;                      // weight rows (2I for gate/up, H for down)
    const uint8_t* a_scales;    // [A][a_sf_stride] E8M0 of the activations
    int a_sf_stride;
    const uint8_t* b_base;      // this layer's slots + offset of the weight matrix
    size_t expert_bytes;
    size_t b_rs;                // bytes per weight row
    int b_code_bytes;           // K/2: scales start here in each row
    int b_sf_bytes;             // pad16(K/32)
    int mode;                   // 0: gate/up -> SwiGLU -> MXFP8 h; 1: down -> weighted combine into out
    int I;                      // mode 0: width of h
    uint8_t* hq;                // mode 0: [A][I]
    uint8_t* hs;                // mode 0: [A][hs_stride]
    int hs_stride;
    const int32_t* perm;        // mode 1: [A] grouped row -> assignment t * k + j
    const float* w;             // mode 1: [A] routing weight of each assignment
    int k;                      // mode 1: assignments per token
    float* out;                 // mode 1: [A / k][N], zero before the launch; w * y added atomically
    int n_group;                // 256-column blocks per tile group (1..NT): the tiles run group by
                                // group, 128-row blocks within a group, columns innermost
    uint32_t* err;              // error bits (device word)
};

struct __align__(1024) Smem {
    uint8_t a[kStages][kStageBytesA];
    uint8_t b[kStages][kStageBytesB];
    uint64_t full[kStages];      // TMA bytes landed
    uint64_t sf_full[2];         // scale factors of a group slot written to tensor memory
    uint64_t sf_empty[2];        // the MMAs of the group that used a slot have finished
    uint64_t empty[kStages];     // MMAs of the stage finished (smem and scale slot free)
    uint64_t acc_full;           // accumulator holds a finished tile
    uint64_t acc_empty;          // epilogue has read the accumulator into registers
    uint64_t mma_done;
    uint32_t tmem_base;
    int32_t mt_prefix[kMaxExperts + 1];  // first 128-row tile of each expert
    int32_t offs[kMaxExperts + 1];       // copy of the group offsets
    int32_t slot[kMaxExperts];           // copy of the slot map
    uint32_t n_tiles;
    // per epilogue warp: 32 rows x 16 fp32 of y, rows padded to 20 words so
    // both the row-wise writes and the column-wise reads are conflict-free
    __align__(16) float ystage[8][32 * kYPad];
};
static_assert(offsetof(Smem, ystage) % 16 == 0 && (32 * kYPad * 4) % 16 == 0, "16-byte staging rows");
static_assert(offsetof(Smem, b) % 1024 == 0 && kStageBytesA % 1024 == 0 && kStageBytesB % 1024 == 0,
              "128-byte-swizzled operand tiles start on 1024-byte boundaries");

struct Tile {
    int e, m0, rows, nt, slot;
};

__device__ __forceinline__ Tile decode_tile(const Smem& sm, const GemmParams& p, int t, int NT) {
    Tile tl;
    int mt;
    const int G = p.n_group;
    if (G >= NT) {
        mt = t / NT;
        tl.nt = t - mt * NT;
    } else {
        // groups of G column blocks (the last one may be narrower)
        const int per = int(sm.n_tiles / uint32_t(NT)) * G;
        const int g = t / per;
        const int r = t - g * per;
        const int Gg = min(G, NT - g * G);
        mt = r / Gg;
        tl.nt = g * G + (r - mt * Gg);
    }
    int lo = 0, hi = p.E;  // largest e with mt_prefix[e] <= mt
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sm.mt_prefix[mid] <= mt) lo = mid; else hi = mid;
    }
    // skip experts with no tiles (equal prefix values)
    while (lo + 1 < p.E && sm.mt_prefix[lo + 1] <= mt) ++lo;
    tl.e = lo;
    tl.m0 = sm.offs[lo] + (mt - sm.mt_prefix[lo]) * kBM;
    tl.rows = min(kBM, sm.offs[lo + 1] - tl.m0);
    tl.slot = sm.slot[lo];
    return tl;
}

constexpr int kRb = kBN / 32;  // 32-row groups of a B tile

// Scale bytes of group g (stages 8g..8g+7, 32 bytes a row) of a tile's
// rows for feeder lane `lane`: A rows m0 + 32c + lane, B rows
// nt * kBN + 32c + lane (clamped to the last row; the clamped rows' factors
// only meet padding), xa[2c + h] / xb[2c + h] the row's h-th 16 bytes;
// zero past the row's scale bytes (a last group of four stages or fewer).
__device__ __forceinline__ void sf_load_group8(const GemmParams& p, const Tile& tl, int lane, int g, uint4 (&xa)[8],
                                               uint4 (&xb)[2 * kRb]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int arow = min(tl.m0 + 32 * c + lane, p.A - 1);
        const uint4* r = reinterpret_cast<const uint4*>(p.a_scales + (size_t)arow * p.a_sf_stride);
#pragma unroll
        for (int h = 0; h < 2; ++h)
            xa[2 * c + h] = (2 * g + h) * 16 < p.a_sf_stride ? __ldg(r + 2 * g + h) : make_uint4(0u, 0u, 0u, 0u);
    }
    const uint8_t* bb = p.b_base + (size_t)tl.slot * p.expert_bytes + p.b_code_bytes;
#pragma unroll
    for (int c = 0; c < kRb; ++c) {
        const int brow = min(tl.nt * kBN + 32 * c + lane, p.N - 1);
        const uint4* r = reinterpret_cast<const uint4*>(bb + (size_t)brow * p.b_rs);
#pragma unroll
        for (int h = 0; h < 2; ++h)
            xb[2 * c + h] = (2 * g + h) * 16 < p.b_sf_bytes ? __ldg(r + 2 * g + h) : make_uint4(0u, 0u, 0u, 0u);
    }
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
    return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// 32 lanes x 16 columns into v[0..15] (v indexes a register array after unrolling).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ float e8m0_inv_scale_f(uint32_t sb) {
    const int ef = 254 - int(sb);
    return ef > 0 ? __uint_as_float(uint32_t(ef) << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ uint32_t e8m0_from_amax(float amax) {
    const uint32_t bits = __float_as_uint(amax);
    const int ef = int((bits >> 23) & 0xffu);
    if (amax == 0.0f || ef == 0) return 0u;
    return uint32_t(min(max(ef - 8, 0), 254));
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                       const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = warp >> 2;
    volatile uint32_t* err = p.err;

    // Programmatic launch hand-off: the next kernel may launch now (its CTAs
    // take SMs as ours exit); this grid reads and writes nothing in global
    // memory before the previous kernel in the stream has finished.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- set-up: tile prefix over experts, barriers, tensor memory ----
    // The offsets and the slot map are copied to shared memory once, so a
    // tile start costs no global-memory round trip in any role.
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < p.E; base += 32) {
            const int e = base + lane;
            int v = 0;
            if (e < p.E) {
                const int o0 = p.offsets[e], o1 = p.offsets[e + 1];
                sm.offs[e] = o0;
                if (e == p.E - 1) sm.offs[p.E] = o1;
                sm.slot[e] = p.slot_of ? p.slot_of[e] : p.slot_tab[e];
                v = (o1 - o0 + kBM - 1) / kBM;
            }
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += u;
            }
            if (e < p.E) sm.mt_prefix[e] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            sm.mt_prefix[p.E] = carry;
            const int NT = (p.N + kBN - 1) / kBN;
            sm.n_tiles = uint32_t(carry) * uint32_t(NT);
            for (int s = 0; s < kStages; ++s) {
                tc::mbar_init(&sm.full[s], 1);
                if (s < 2) {
                    tc::mbar_init(&sm.sf_full[s], 128);
                    tc::mbar_init(&sm.sf_empty[s], 1);
                }
                tc::mbar_init(&sm.empty[s], 1);
            }
            tc::mbar_init(&sm.acc_full, 1);
            tc::mbar_init(&sm.acc_empty, 256);
            tc::mbar_init(&sm.mma_done, 1);
            tc::fence_barrier_init();
            tc::tma_prefetch_desc(&map_a);
            tc::tma_prefetch_desc(&map_b);
        }
    } else if (warp == 1) {
        tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const int NT = (p.N + kBN - 1) / kBN;
    const int n_tiles = int(sm.n_tiles);
    const int n_kstages = (p.K + kBK - 1) / kBK;

    if (wg == 0) {
        setmaxnreg_dec<kRegsCtl>();
        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            for (int t = blockIdx.x; t < n_tiles && !*err; t += gridDim.x) {
                const Tile tl = decode_tile(sm, p, t, NT);
                const int slot = tl.slot;
                if (slot < 0 || slot >= p.S) {
                    atomicOr(const_cast<uint32_t*>(err), 4u);
                    break;
                }
                for (int ks = 0; ks < n_kstages; ++ks) {
                    if (!tc::mbar_wait_hot(&sm.empty[stage], phase ^ 1u, err, 1u)) break;
                    tc::mbar_arrive_expect_tx(&sm.full[stage], kStageBytesA + kTxBytesB);
                    tc::tma_load_2d(sm.a[stage], &map_a, &sm.full[stage], ks * kBK, tl.m0);
                    tc::tma_load_3d(sm.b[stage], &map_b, &sm.full[stage], ks * kBK, tl.nt * kBN, slot);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
        } else if (warp == 1 && lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0;
            uint32_t phase = 0;
            int i = 0;
            int gr = 0;   // scale-factor groups consumed so far
            for (int t = blockIdx.x; t < n_tiles && !*err; t += gridDim.x, ++i) {
                // the epilogue has read tile i - 1 out of the accumulator
                if (!tc::mbar_wait_hot(&sm.acc_empty, (i & 1) ^ 1u, err, 2u)) break;
                tc::tc_fence_after();
                bool ok = true;
                for (int ks = 0; ks < n_kstages; ++ks) {
                    const int sg = ks & (kSfGroup - 1);
                    if ((sg == 0 && !tc::mbar_wait_hot(&sm.sf_full[gr & 1], uint32_t(gr >> 1) & 1u, err, 2u)) ||
                        !tc::mbar_wait_hot(&sm.full[stage], phase, err, 2u)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(sm.a[stage]);
                    const uint32_t b0 = tc::smem_u32(sm.b[stage]);
                    const uint32_t sfa = tmem + sf_col_g(gr & 1, sg);
#pragma unroll
                    for (int kk = 0; kk < kBK / 32; ++kk) {
                        const int kb = ks * (kBK / 32) + kk;
                        if (kb < p.KB) {
                            const uint32_t idesc = tc::idesc_mxf8f6f4(0, 5, kBM, kBN, kk, kk);
                            tc::mma_mxf8f6f4(tmem, tc::smem_desc_sw128(a0 + kk * 32),
                                             tc::smem_desc_sw128(b0 + kk * 32), idesc, sfa, sfa + 8,
                                             (ks | kk) != 0);
                        }
                    }
                    tc::mma_commit(&sm.empty[stage]);
                    if (sg == kSfGroup - 1 || ks == n_kstages - 1) {
                        tc::mma_commit(&sm.sf_empty[gr & 1]);
                        ++gr;
                    }
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc::mma_commit(&sm.acc_full);
            }
            // all MMAs issued by this CTA have finished before TMEM is freed
            tc::mma_commit(&sm.mma_done);
            tc::mbar_wait(&sm.mma_done, 0, err, 16u);
        }
    } else if (wg == 1) {
        setmaxnreg_inc<kRegsSf>();
        // ---------------- scale-factor feeders (warps 4..7 = lane quarters 0..3) ----------------
        // Thread (quarter q, lane l) writes lane 32q + l of a group slot:
        // for each stage of the group, column c of the A part gets the
        // stage's four scale bytes of activation row 32c + l (c < 4), column
        // c of the B part those of weight row 32c + l (c < kBN / 32).  Each
        // row's bytes are read 32 at a time (a group of eight stages) right
        // after the previous group is written, a group ahead of their use --
        // across tile boundaries too, so a new tile's first stages never
        // wait for loads; one register set suffices.
        const int q = warp & 3;
        const uint32_t lane_base = tmem + (uint32_t(q * 32) << 16);
        const int ngroups = (n_kstages + kSfGroup - 1) / kSfGroup;
        int gr = 0;   // scale-factor groups written so far
        int t = blockIdx.x;
        Tile tl{};
        uint4 xa[8], xb[2 * kRb];
        bool have = false;
        if (t < n_tiles) {
            tl = decode_tile(sm, p, t, NT);
            if (tl.slot >= 0 && tl.slot < p.S) {
                sf_load_group8(p, tl, lane, 0, xa, xb);
                have = true;
            }
        }
        while (have && !*err) {
            const int tn = t + gridDim.x;
            Tile nx{};
            bool next_ok = false, ok = true;
            for (int g = 0; g < ngroups && ok; ++g) {
                // the group slot is free once the MMAs of the group two back have finished
                if (gr >= 2 && !tc::mbar_wait_hot(&sm.sf_empty[gr & 1], uint32_t((gr >> 1) + 1) & 1u, err, 64u)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
#pragma unroll
                for (int w = 0; w < kSfGroup; ++w) {
                    if (kSfGroup * g + w >= n_kstages) break;
                    const uint32_t col = lane_base + sf_col_g(gr & 1, w);
                    const int h = w >> 2, wi = w & 3;
                    tc::tmem_st_x4(col, word_of(xa[h], wi), word_of(xa[2 + h], wi), word_of(xa[4 + h], wi),
                                   word_of(xa[6 + h], wi));
                    uint32_t bw[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) bw[c] = c < kRb ? word_of(xb[2 * (c < kRb ? c : 0) + h], wi) : 0u;
                    tc::tmem_st_x8(col + 8, bw);
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                tc::mbar_arrive(&sm.sf_full[gr & 1]);
                ++gr;
                // the next group's bytes, loaded while this group is consumed
                if (g + 1 < ngroups) {
                    sf_load_group8(p, tl, lane, g + 1, xa, xb);
                } else if (tn < n_tiles) {
                    nx = decode_tile(sm, p, tn, NT);
                    next_ok = nx.slot >= 0 && nx.slot < p.S;
                    if (next_ok) sf_load_group8(p, nx, lane, 0, xa, xb);
                }
            }
            if (!ok || !next_ok) break;
            t = tn;
            tl = nx;
        }
    } else {
        setmaxnreg_inc<kRegsEpi>();
        // ---------------- epilogue (warps 8..15) ----------------
        // Warp w serves lane quarter w % 4 (tile rows) and half (w - 8) / 4
        // of the tile's columns.  It copies its 32 rows x kBN/2 columns of
        // the accumulator into registers, releases the accumulator to the
        // next tile's MMAs, and finishes the tile from registers.
        constexpr int kHalf = kBN / 2;
        const int q = warp & 3, hh = wg - 2;
        const int r = q * 32 + lane;                // tile row == TMEM lane
        const uint32_t lane_base = tmem + (uint32_t(q * 32) << 16) + uint32_t(hh * kHalf);
        int i = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
            if (*err) break;
            const Tile tl = decode_tile(sm, p, t, NT);
            // mode 1: the token and routing weight of the four tile rows this
            // thread stores, fetched before the accumulator is ready
            int tok[4] = {-1, -1, -1, -1};
            float wgt[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (p.mode != 0) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int row = q * 32 + (lane >> 2) + 8 * j;
                    const int mm = tl.m0 + row;
                    if (row < tl.rows && mm < p.A) {
                        const int a = __ldg(p.perm + mm);
                        if (a >= 0 && a < p.A) {
                            tok[j] = a / p.k;
                            wgt[j] = __ldg(p.w + a);
                        }
                    }
                }
            }
            if (!tc::mbar_wait(&sm.acc_full, i & 1, err, 8u)) break;
            tc::tc_fence_after();
            uint32_t v[kHalf];
#pragma unroll
            for (int c = 0; c < kHalf / 16; ++c) tmem_ld16(lane_base + 16 * c, &v[16 * c]);
            tc::tmem_ld_wait();
            tc::tc_fence_before();
            tc::mbar_arrive(&sm.acc_empty);
            const bool valid = r < tl.rows;
            const int m = tl.m0 + r;
            if (p.mode == 0) {
                // columns 64j..64j+31 of the tile: gate rows of chunk c = (kBN/64) nt + j
                // (h columns 32c..32c+31); 64j+32..64j+63: the matching up rows
#pragma unroll
                for (int jj = 0; jj < kHalf / 64; ++jj) {
                    const int chunk = tl.nt * (kBN / 64) + hh * (kHalf / 64) + jj;
                    if (chunk * 32 >= p.I) break;   // ragged last tile (warp-uniform)
                    float hv[32];
                    float amax = 0.0f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float g = __uint_as_float(v[64 * jj + j]);
                        const float u = __uint_as_float(v[64 * jj + 32 + j]);
                        const float s = g / (1.0f + expf(-g));
                        const float hb = __bfloat162float(__float2bfloat16_rn(s * u));
                        hv[j] = hb;
                        amax = fmaxf(amax, fabsf(hb));
                    }
                    if (valid) {
                        const uint32_t sb = e8m0_from_amax(amax);
                        const float mul = e8m0_inv_scale_f(sb);
                        uint32_t wv[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            wv[j] = cvt_e4m3x2(hv[4 * j] * mul, hv[4 * j + 1] * mul) |
                                    (cvt_e4m3x2(hv[4 * j + 2] * mul, hv[4 * j + 3] * mul) << 16);
                        const int col = chunk * 32;
                        uint4* dst = reinterpret_cast<uint4*>(p.hq + (size_t)m * p.I + col);
                        if ((reinterpret_cast<uintptr_t>(dst) & 15) != 0 || m >= p.A || col + 32 > p.I) {
                            atomicOr(const_cast<uint32_t*>(err), 32u);
                        } else {
                            dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                            dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
                            p.hs[(size_t)m * p.hs_stride + col / 32] = uint8_t(sb);
                        }
                    }
                }
            } else {
                // y rows leave through a per-warp shared tile so that one
                // vector atomic instruction covers 64 contiguous bytes in each
                // of 8 output rows instead of 16 bytes in each of 32 rows; the
                // k assignments of a token land in out[token] in whatever
                // order their tiles finish (fp32 atomics).
                float* st = sm.ystage[warp - 8];
                const int rr0 = lane >> 2, qq = lane & 3;
#pragma unroll
                for (int c = 0; c < kHalf / 16; ++c) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<float4*>(st + lane * kYPad + 4 * j) =
                            make_float4(__uint_as_float(v[16 * c + 4 * j]), __uint_as_float(v[16 * c + 4 * j + 1]),
                                        __uint_as_float(v[16 * c + 4 * j + 2]),
                                        __uint_as_float(v[16 * c + 4 * j + 3]));
                    __syncwarp();
                    const int n = tl.nt * kBN + hh * kHalf + c * 16 + 4 * qq;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int rr = rr0 + 8 * j;              // row within this warp's 32
                        const float4 val = *reinterpret_cast<const float4*>(st + rr * kYPad + 4 * qq);
                        if (tok[j] >= 0 && n < p.N) {
                            float4* dst = reinterpret_cast<float4*>(p.out + (size_t)tok[j] * p.N + n);
                            if ((reinterpret_cast<uintptr_t>(dst) & 15) != 0)
                                atomicOr(const_cast<uint32_t*>(err), 32u);
                            else
                                atomicAdd(dst, make_float4(wgt[j] * val.x, wgt[j] * val.y, wgt[j] * val.z,
                                                           wgt[j] * val.w));
                        }
                    }
                    __syncwarp();
                }
            }
        }
    }

    // ---- teardown: every role has left its loop ----
    __syncthreads();
    if (*err && threadIdx.x == 0) {
        // after a failure, give tile copies already issued time to land
        // before the CTA's shared memory is released
        for (int i = 0; i < 2000; ++i) __nanosleep(100);
    }
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- host side -------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int get_encoder(EncodeTiledFn* out) {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    static cudaError_t status = cudaSuccess;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (status == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!fn) return status != cudaSuccess ? cuda_fail(status) : MOE_ERR_UNSUPPORTED;
    *out = fn;
    return MOE_OK;
}

// Activation rows: [rows][K] bytes (E4M3), tile 128 x 128.
int make_map_act(CUtensorMap* m, const void* base, int K, int rows) {
    EncodeTiledFn enc = nullptr;
    int rc = get_encoder(&enc);
    if (rc != MOE_OK) return rc;
    const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(K)};
    const cuuint32_t box[2] = {uint32_t(kBK), uint32_t(kBM)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

// Weight rows of every slot of a layer: [S][rows][row_bytes] with K E2M1
// codes at the start of each row, unpacked by TMA into 16-byte-aligned
// groups of 16.  The inner extent is K rounded up to 128 (a TMA rule for
// this type); the extra codes come from the row's own scale bytes and are
// never multiplied (the MMA loop stops at K).
int make_map_weights(CUtensorMap* m, const void* base, int K, int rows, int slots, size_t row_bytes,
                     size_t expert_bytes) {
    EncodeTiledFn enc = nullptr;
    int rc = get_encoder(&enc);
    if (rc != MOE_OK) return rc;
    const size_t k128 = round_up(size_t(K), 128);
    if (k128 / 2 > row_bytes || (reinterpret_cast<uintptr_t>(base) & 31)) return MOE_ERR_UNSUPPORTED;
    const cuuint64_t dims[3] = {cuuint64_t(k128), cuuint64_t(rows), cuuint64_t(slots)};
    const cuuint64_t strides[2] = {cuuint64_t(row_bytes), cuuint64_t(expert_bytes)};
    const cuuint32_t box[3] = {uint32_t(kBK), uint32_t(kBN), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

size_t smem_bytes() { return sizeof(Smem) + 1024; }

int launch_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const GemmParams& p, int max_tiles, cudaStream_t s) {
    static DeviceOnce attr_set;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != MOE_OK) return rc;
    if (di.cc_major < 10) return MOE_ERR_UNSUPPORTED;
    if (smem_bytes() > di.smem_optin) return MOE_ERR_UNSUPPORTED;
    if (di.device < 0 || di.device >= 64) return MOE_ERR_UNSUPPORTED;
    if (!attr_set.done(di.device)) {
        // The warpgroups' register split must add up to exactly what the
        // launch grants each thread, or a setmaxnreg.inc would wait forever.
        cudaFuncAttributes fa{};
        MOE_CUDA_TRY(cudaFuncGetAttributes(&fa, grouped_gemm_tc_kernel));
        if (fa.numRegs != kLaunchRegs || fa.maxThreadsPerBlock < kThreads) return MOE_ERR_UNSUPPORTED;
        MOE_CUDA_TRY(cudaFuncSetAttribute(grouped_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem_bytes()));
        attr_set.mark(di.device);
    }
    const int grid = max(1, min(di.sms, max_tiles));
    // programmatic stream serialisation (the kernel waits for its
    // predecessor with griddepcontrol before touching global memory)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(unsigned(kThreads));
    cfg.dynamicSmemBytes = smem_bytes();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, grouped_gemm_tc_kernel, ma, mb, p));
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

struct PrefillWs {
    size_t xq, xs, hq, hs, err, total;
    int xs_stride, hs_stride;
};

PrefillWs prefill_ws(int T, int k, int H, int I) {
    PrefillWs w;
    const size_t A = size_t(T) * k;
    w.xs_stride = int(pad16(size_t(H) / 32));
    w.hs_stride = int(pad16(size_t(I) / 32));
    size_t o = 0;
    w.err = o; o += 256;
    w.xq = o; o = round_up(o + A * H, 256);
    w.xs = o; o = round_up(o + A * w.xs_stride, 256);
    w.hq = o; o = round_up(o + A * I, 256);
    w.hs = o; o = round_up(o + A * w.hs_stride, 256);
    w.total = o;
    return w;
}

}  // namespace

size_t prefill_workspace_bytes(int T, int k, int H, int I) { return prefill_ws(T, k, H, I).total; }

// Zero the error word, scale buffers and out; quantise every token's x once
// into its k grouped rows.
int launch_prefill_prepare(const FfnArgs& a, void* ws, size_t ws_bytes, cudaStream_t s) {
    const Layout& L = *a.L;
    const PrefillWs w = prefill_ws(a.T, a.k, L.H, L.I);
    if (ws_bytes < w.total) return MOE_ERR_INVALID;
    if (L.H > 4096 || L.I > 4096 || a.E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
    if (a.T == 0) return MOE_OK;
    const int A = a.T * a.k;
    uint8_t* base = static_cast<uint8_t*>(ws);
    MOE_CUDA_TRY(cudaMemsetAsync(base + w.err, 0, 4, s));
    MOE_CUDA_TRY(cudaMemsetAsync(base + w.xs, 0, size_t(A) * w.xs_stride, s));
    MOE_CUDA_TRY(cudaMemsetAsync(base + w.hs, 0, size_t(A) * w.hs_stride, s));
    if (!a.accumulate) MOE_CUDA_TRY(cudaMemsetAsync(a.out, 0, size_t(a.T) * L.H * sizeof(float), s));
    return launch_quant_mxfp8_scatter(a.x, L.H, a.inv, a.k, a.T, base + w.xq, base + w.xs, w.xs_stride, s);
}

// Gate/up and down GEMMs over the groups of experts [e0, e1); the down
// epilogue adds w * y into out.  Slots come from slot_tab (host, e1 - e0
// entries) when given, else from the device map a.slot_of.  max_mtiles
// bounds the 128-row tiles of those groups (it only sizes the grid).
int launch_prefill_experts(const FfnArgs& a, void* ws, int e0, int e1, const int32_t* slot_tab, int max_mtiles,
                           cudaStream_t s) {
    const Layout& L = *a.L;
    const PrefillWs w = prefill_ws(a.T, a.k, L.H, L.I);
    if (e0 < 0 || e1 > a.E || e0 > e1) return MOE_ERR_INVALID;
    if (slot_tab && e1 - e0 > kMaxSlotTab) return MOE_ERR_UNSUPPORTED;
    if (a.T == 0 || e0 == e1 || max_mtiles <= 0) return MOE_OK;
    const int A = a.T * a.k;
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint8_t* xq = base + w.xq;
    uint8_t* xs = base + w.xs;
    uint8_t* hq = base + w.hq;
    uint8_t* hs = base + w.hs;
    uint32_t* err = reinterpret_cast<uint32_t*>(base + w.err);

    CUtensorMap map_x, map_gu, map_h, map_d;
    int rc = make_map_act(&map_x, xq, L.H, A);
    if (rc == MOE_OK) rc = make_map_weights(&map_gu, a.slots, L.H, 2 * L.I, a.S, L.rs_gu, a.expert_bytes);
    if (rc == MOE_OK) rc = make_map_act(&map_h, hq, L.I, A);
    if (rc == MOE_OK) rc = make_map_weights(&map_d, a.slots + L.d_off, L.I, L.H, a.S, L.rs_d, a.expert_bytes);
    if (rc != MOE_OK) return rc;

    GemmParams g{};
    g.offsets = a.offsets + e0;
    g.E = e1 - e0;
    if (slot_tab) {
        g.slot_of = nullptr;
        for (int e = 0; e < g.E; ++e) g.slot_tab[e] = slot_tab[e];
    } else {
        g.slot_of = a.slot_of + e0;
    }
    g.A = A;
    g.S = a.S;
    g.expert_bytes = a.expert_bytes;
    g.err = err;
    // gate/up: K = H, N = 2I, epilogue SwiGLU -> MXFP8 h
    g.K = L.H;
    g.KB = L.H / 32;
    g.N = 2 * L.I;
    g.a_scales = xs;
    g.a_sf_stride = w.xs_stride;
    g.b_base = a.slots;
    g.b_rs = L.rs_gu;
    g.b_code_bytes = L.H / 2;
    g.b_sf_bytes = int(pad16(size_t(L.H) / 32));
    g.mode = 0;
    g.I = L.I;
    g.hq = hq;
    g.hs = hs;
    g.hs_stride = w.hs_stride;
    g.n_group = (g.N + kBN - 1) / kBN;
    rc = launch_gemm(map_x, map_gu, g, max_mtiles * ((g.N + kBN - 1) / kBN), s);
    if (rc != MOE_OK) return rc;
    // down: K = I, N = H, epilogue w * y added into out[token]
    g.K = L.I;
    g.KB = L.I / 32;
    g.N = L.H;
    g.a_scales = hs;
    g.a_sf_stride = w.hs_stride;
    g.b_base = a.slots + L.d_off;
    g.b_rs = L.rs_d;
    g.b_code_bytes = L.I / 2;
    g.b_sf_bytes = int(pad16(size_t(L.I) / 32));
    g.mode = 1;
    g.perm = a.perm;
    g.w = a.w;
    g.k = a.k;
    g.out = a.out;
    // The down tiles of one column block add into that block of every
    // routed token's row of out: when out is larger than half of L2, the
    // tiles run a few column blocks at a time so that the out rows they
    // read-modify-write stay in L2.
    {
        const int NT = (g.N + kBN - 1) / kBN;
        const size_t per_block = size_t(a.T) * kBN * sizeof(float);
        const size_t budget = size_t(64) << 20;
        g.n_group = size_t(a.T) * size_t(g.N) * sizeof(float) <= budget
                        ? NT
                        : int(std::max<size_t>(1, std::min<size_t>(size_t(NT), budget / per_block)));
    }
    return launch_gemm(map_h, map_d, g, max_mtiles * ((g.N + kBN - 1) / kBN), s);
}

int launch_prefill_ffn(const FfnArgs& a, void* ws, size_t ws_bytes, cudaStream_t s) {
    int rc = launch_prefill_prepare(a, ws, ws_bytes, s);
    if (rc != MOE_OK || a.T == 0) return rc;
    return launch_prefill_experts(a, ws, 0, a.E, nullptr, a.T * a.k / kBM + a.E, s);
}

}  // namespace moe
