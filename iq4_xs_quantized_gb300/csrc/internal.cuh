// internal.cuh -- layout constants, decoders and PTX wrappers shared by the
// kernels of libiq4xs.so.  Not part of the public ABI (include/iq4xs.h).
//
// Format facts (V100TPS engine page, agent-report.daedalus.work/V100TPS/
// engine.html, tile-geometry passage after the new-kernel table): an IQ4_XS
// sub-block of 32 weights is 4 ints of packed nibbles, low nibbles are
// elements 0-15 and high nibbles 16-31; its scale is d*(ls-32); a nibble is
// decoded through kvalues_iq4nl.  The same passage records that reusing
// thread-mapping constants as tile geometry silently advanced four
// super-blocks per step, so every tile size here is a named constant tied to
// the format by static_assert.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace iq4xs {

// ---------------------------------------------------------------------------
// IQ4_XS super-block and Q8_1 block.
// ---------------------------------------------------------------------------
constexpr int kQK = 256;                      // weights per super-block
constexpr int kSub = 32;                      // weights per sub-block == per Q8_1 block
constexpr int kSubPerBlock = kQK / kSub;      // 8
constexpr int kBlockBytes = 136;              // 2 + 2 + 4 + 128
constexpr int kQsBytesPerSub = kSub / 2;      // 16 bytes of nibbles per sub-block

struct BlockIQ4XS {
    uint16_t d;            // fp16 super-block scale
    uint16_t scales_h;     // 2 high bits of each ls_j at bits 2j..2j+1
    uint8_t scales_l[4];   // 4 low bits of ls_j: low nibble for even j, high for odd j
    uint8_t qs[kQK / 2];   // nibbles; sub-block j uses bytes 16j..16j+15
};
static_assert(sizeof(BlockIQ4XS) == kBlockBytes, "IQ4_XS super-block is 136 bytes");
static_assert(offsetof(BlockIQ4XS, d) == 0, "d at byte 0");
static_assert(offsetof(BlockIQ4XS, scales_h) == 2, "scales_h at byte 2");
static_assert(offsetof(BlockIQ4XS, scales_l) == 4, "scales_l at byte 4");
static_assert(offsetof(BlockIQ4XS, qs) == 8, "qs at byte 8");
static_assert(kSubPerBlock * kQsBytesPerSub == sizeof(((BlockIQ4XS*)0)->qs), "8 sub-blocks of 16 bytes");

constexpr int kQ8Max = 127;  // Q8_1 codes lie in [-127, 127]

// ---------------------------------------------------------------------------
// Weight formats.  The same engine page's tile-geometry passage: an IQ4_XS
// sub-block is exactly one Q4_0 block (16 bytes of nibbles, low nibbles
// elements 0-15, high nibbles 16-31); only the scale (one fp16 d per 32
// weights for Q4_0, d*(ls-32) for IQ4_XS) and the nibble's value (q-8 for
// Q4_0, kvalues_iq4nl for IQ4_XS) differ.  IQ4_NL is kvalues_iq4nl on
// 32-weight blocks of 18 bytes (forum page on the Qwen3.5 engine: the
// (32, 18) block shape).  Q4_0 and IQ4_NL share one byte shape: fp16 d at
// byte 0, nibbles at bytes 2..17.  Every format's row is a whole number of
// 256-weight groups here (136 or 8 x 18 = 144 bytes), so rows stay 16-byte
// aligned and a 32-weight block starts 2 bytes past a 4-byte boundary
// exactly when its index is odd.
// ---------------------------------------------------------------------------
enum WType : int { kWtIQ4XS = 0, kWtQ4_0 = 1, kWtIQ4NL = 2 };
constexpr int kB18Bytes = 18;                      // one Q4_0 / IQ4_NL block
constexpr int kB18GroupBytes = kSubPerBlock * kB18Bytes;  // 144 per 256 weights
static_assert(kB18GroupBytes % 16 == 0, "256-weight groups of 18-byte blocks keep rows 16-byte aligned");
__host__ __device__ constexpr int wt_group_bytes(int wt) {
    return wt == kWtIQ4XS ? kBlockBytes : kB18GroupBytes;
}
__host__ __device__ inline int64_t wt_row_bytes(int wt, int64_t K) {
    return (K / kQK) * wt_group_bytes(wt);
}

// kvalues_iq4nl packed four entries per word, little endian (entry 4w+k in
// byte k of word w).  Two forms: the int8 values themselves, and u = kv + 128
// (all of 1..241 fit one unsigned byte) for building exact fp16 operands.
constexpr uint32_t kKvS8_0 = 0xBFAD9881u, kKvS8_1 = 0xF6EADDCFu, kKvS8_2 = 0x26190D01u,
                   kKvS8_3 = 0x71594535u;
constexpr uint32_t kKvU8_0 = 0x3F2D1801u, kKvU8_1 = 0x766A5D4Fu, kKvU8_2 = 0xA6998D81u,
                   kKvU8_3 = 0xF1D9C5B5u;
// Q4_0's nibble values q-8, in the same two forms (int8; u = q-8+128).
__host__ __device__ constexpr uint32_t q4_0_word(int w, int bias) {
    return (uint32_t)((4 * w + 0 - 8 + bias) & 0xFF) | ((uint32_t)((4 * w + 1 - 8 + bias) & 0xFF) << 8) |
           ((uint32_t)((4 * w + 2 - 8 + bias) & 0xFF) << 16) | ((uint32_t)((4 * w + 3 - 8 + bias) & 0xFF) << 24);
}
// fp16 with bit pattern 0x64XX is 1024 + XX; 1024 + u - 1152 = value exactly.
constexpr uint32_t kF16HiByte = 0x64646464u;
constexpr uint32_t kF16Offset2 = 0x64806480u;  // half2(1152, 1152)

// Nibble-value tables of a format: T8 the int8 values, TU the u = value+128 bytes.
template <int WT>
struct WTables {
    static constexpr uint32_t S0 = kKvS8_0, S1 = kKvS8_1, S2 = kKvS8_2, S3 = kKvS8_3;
    static constexpr uint32_t U0 = kKvU8_0, U1 = kKvU8_1, U2 = kKvU8_2, U3 = kKvU8_3;
};
template <>
struct WTables<kWtQ4_0> {
    static constexpr uint32_t S0 = q4_0_word(0, 0), S1 = q4_0_word(1, 0), S2 = q4_0_word(2, 0),
                              S3 = q4_0_word(3, 0);
    static constexpr uint32_t U0 = q4_0_word(0, 128), U1 = q4_0_word(1, 128),
                              U2 = q4_0_word(2, 128), U3 = q4_0_word(3, 128);
};
static_assert(WTables<kWtQ4_0>::S0 == 0xFBFAF9F8u && WTables<kWtQ4_0>::S3 == 0x07060504u,
              "Q4_0 values -8..7 as int8");
static_assert(WTables<kWtQ4_0>::U0 == 0x7B7A7978u && WTables<kWtQ4_0>::U3 == 0x87868584u,
              "Q4_0 values + 128");

// ---------------------------------------------------------------------------
// Tensor-core path geometry.
// ---------------------------------------------------------------------------
constexpr int kTileN = 128;                       // W rows per CTA = TMEM lanes = UMMA M
constexpr int kPairBlocks = 2;                    // super-blocks per W stage
constexpr int kPairK = kPairBlocks * kQK;         // 512
constexpr int kPairBytes = kPairBlocks * kBlockBytes;  // 272 = 17 x 16: TMA rows stay 16-byte aligned
constexpr int kSubPerPair = kPairK / kSub;        // 16
static_assert(kPairBytes % 16 == 0, "a W stage row must be a whole number of 16-byte units");
static_assert(kPairBytes / 4 <= 256, "TMA box inner extent (uint32 elements) <= 256");
constexpr int kChunkElems = 8;                    // fp16 per 16-byte core-matrix row
constexpr int kChunksPerSub = kSub / kChunkElems; // 4
constexpr int kUmmaK = 16;                        // K per tcgen05.mma kind::f16
constexpr int kMmaPerSub = kSub / kUmmaK;         // 2
constexpr int kASubBytes = kTileN * kSub * 2;     // 8 KB of fp16 A per sub-block
constexpr int kBStageSubs = 4;                    // sub-blocks per activation stage
constexpr int kBStageChunks = kBStageSubs * kChunksPerSub;  // 16
constexpr int kMaxMTile = 128;                    // activation rows per tcgen05 tile (UMMA N)
static_assert(kSubPerPair % kBStageSubs == 0, "activation stages tile a W stage");

// Activation tile height for a batch of M rows: round M up to 16 (UMMA N
// granularity for M=128), capped at kMaxMTile.
__host__ __device__ inline int tc_mtile(int64_t M) {
    int64_t r = (M + 15) / 16 * 16;
    return (int)(r < kMaxMTile ? r : kMaxMTile);
}
__host__ __device__ inline int64_t tc_num_mtiles(int64_t M) {
    int mt = tc_mtile(M);
    return (M + mt - 1) / mt;
}
// Prepared tensor-core operand (written by the quantizer on request, for the
// faster form of the tensor-core matmul): the dequantized activations
// v = q*d_h (d_h the block's stored fp16 scale), times a power of two 2^-e
// per row and span of kScaleSpan values, as a pair of fp16 values hi + lo:
// hi = fp16(v*2^-e), lo = fp16(v*2^-e - hi).  q has 8 significant bits and
// d_h 11, so v has at most 19 and the pair holds it exactly (lo keeps the low
// 8 bits) whenever v*2^-e is a multiple of 2^-24.  e is the smallest e >= 0
// with 127 * max_span(d_h) * 2^-e < 65504: hi never overflows, e = 0 (every
// value exact) unless the span's values reach the fp16 range, and otherwise
// only blocks 2^14 times smaller than the span's largest lose low bits.  The
// matmul scales its fp32 partial sums by 2^e (exact) per span.  With d_x
// folded into the operand the kernel does no per-CTA conversion and its
// epilogue one FMA per element (the Q8_1 form: two FP operations and a scale
// load), for two MMAs more per sub-block.
//   planes: [mtile][K/32 sub-block][plane hi, lo][4 chunks of 8 K][MT rows][8 fp16]
//           (16 B per (chunk, row); a sub-block is 8*MT*16 bytes)
//   then:   [mtile][ceil(K/kScaleSpan) span][MT rows] fp32 2^e
// K is permuted within every sub-block as in the Q8_1 form (below).
constexpr int kPlanes = 2;  // hi, lo
__host__ __device__ inline int64_t tc_qh_bytes(int64_t M, int64_t K) {
    return tc_num_mtiles(M) * (int64_t)tc_mtile(M) * K * 2 * kPlanes;
}
constexpr int kScaleSpan = 1024;                  // values per activation scale span
constexpr int kSubPerSpan = kScaleSpan / kSub;     // 32 sub-blocks
__host__ __device__ inline int64_t tc_num_spans(int64_t K) { return (K + kScaleSpan - 1) / kScaleSpan; }
__host__ __device__ inline int64_t tc_operand_total_bytes(int64_t M, int64_t K) {
    return tc_qh_bytes(M, K) + tc_num_mtiles(M) * tc_num_spans(K) * (int64_t)tc_mtile(M) * 4;
}

// Activation operand of the tensor-core path in its Q8_1 form, built inside
// the matmul from the Q8_1 codes: each code q (|q| <= 127) as an exact fp16 integer, in the
// K order of the decoded weights.  Within every sub-block K position 2i+h
// holds element i+16h (one qs byte decodes to elements i and 16+i), so a
// 16-byte chunk c (K positions 8c..8c+7) holds elements
// (4c, 16+4c, 4c+1, 16+4c+1, ..., 4c+3, 16+4c+3).
//   per sub-block: [4 chunks of 8 K][MT rows][8 fp16]  (16 B per (chunk, row))
// The products kv*q are integers of magnitude <= 127*127 and a sub-block's
// sum of 32 is at most 516,128 < 2^24, so the fp32 accumulator holds the
// exact integer dot of the sub-block, whatever the summation order.
constexpr int kQRowBytes = kBStageSubs * kSub;  // Q8_1 codes of one row per activation stage
static_assert(kQRowBytes == 128, "one 128-byte swizzle row per activation row and stage");

// Eight Q8_1 codes -> the 16-byte fp16 chunk above.  lo4 holds elements
// 4c..4c+3 (one byte each), hi4 elements 16+4c..16+4c+3.  fp16 with bit
// pattern 0x64XX is 1024 + XX, and q ^ 0x80 is q + 128 as an unsigned byte,
// so each half is (1152 + q) - 1152 = q exactly.
__device__ __forceinline__ uint4 q8x8_to_f16(uint32_t lo4, uint32_t hi4) {
    const uint32_t ua = lo4 ^ 0x80808080u, ub = hi4 ^ 0x80808080u;
    const uint32_t p01 = __byte_perm(ua, ub, 0x5140u);  // [a0, b0, a1, b1]
    const uint32_t p23 = __byte_perm(ua, ub, 0x7362u);  // [a2, b2, a3, b3]
    const uint32_t w[4] = {__byte_perm(p01, 0x64646464u, 0x4140u), __byte_perm(p01, 0x64646464u, 0x4342u),
                           __byte_perm(p23, 0x64646464u, 0x4140u), __byte_perm(p23, 0x64646464u, 0x4342u)};
    const uint32_t off_bits = 0x64806480u;  // half2(1152, 1152)
    const __half2 off = *reinterpret_cast<const __half2*>(&off_bits);
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&w[k]), off);
        o[k] = *reinterpret_cast<uint32_t*>(&v);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------------------
// Device error word (defined in api.cu); its address is passed to kernels.
// ---------------------------------------------------------------------------
enum DeviceError : int {
    kDevErrNone = 0,
    kDevErrTimeoutW = 0x101,
    kDevErrTimeoutB = 0x102,
    kDevErrTimeoutA = 0x103,
    kDevErrTimeoutMma = 0x104,
    kDevErrTimeoutFree = 0x105,
    kDevErrTimeoutDrain = 0x106,
    kDevErrTimeoutRecv = 0x107,
    kDevErrTimeoutQ = 0x108,
    kDevErrTimeoutX = 0x109,
    kDevErrLayout = 0x10A,  // dynamic shared memory not 1024-byte aligned
    kDevErrTimeoutMmaStage = 0x10B,  // warp-MMA matmul: a stage (W and codes) never landed
    kDevErrTimeoutMmaSlot = 0x10C,   // warp-MMA matmul: a stage slot was never freed
    kDevErrBounds = 0x200,           // + BoundsSite: a checked access missed its buffer
};

// ---------------------------------------------------------------------------
// Bounds-checked debug build (compiled with -DIQ4XS_BOUNDS_CHECK into a
// library of its own).  Every plain global access of a kernel, every TMA box
// origin and every computed shared-memory offset is checked against the
// extent the kernel derives from its own arguments.  A miss records
// kDevErrBounds + site in the device error word (the first code recorded
// sticks) and skips the access: a load yields zero, a store is dropped.  A
// TMA box origin outside its tensor is recorded only (the copy unit fills
// such boxes itself); an innermost coordinate off the 16-byte grid is
// recorded and its copy skipped (the stage's bounded wait then runs out
// instead of the copy faulting).  The 8 bytes at word 2 of the error array
// hold a margin subtracted from every global extent, so that in-range
// accesses within that many bytes of a buffer's end are reported although no
// access leaves the buffer.  In the normal build every check is the constant
// true and compiles away.
// ---------------------------------------------------------------------------
enum BoundsSite : int {
    kBcQuantX = 1, kBcQuantQs, kBcQuantDs, kBcQuantOp, kBcQuantSpan,
    kBcDqW = 0x10, kBcDqOut,
    kBcDp4aW = 0x20, kBcDp4aQs, kBcDp4aDs, kBcDp4aY, kBcDp4aOffsets, kBcDp4aRows,
    kBcMmaW = 0x30, kBcMmaWAlign, kBcMmaQ, kBcMmaQAlign, kBcMmaDs, kBcMmaY, kBcMmaOffsets,
    kBcMmaRows, kBcMmaSmem, kBcMmaSplit,
    kBcTcW = 0x40, kBcTcWAlign, kBcTcQ, kBcTcQAlign, kBcTcOp, kBcTcDs, kBcTcY, kBcTcSpan,
    kBcTcSmem, kBcTcRecv, kBcTcRows,
};
#ifdef IQ4XS_BOUNDS_CHECK
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif
constexpr int kErrWords = 4;  // error code, spare, 64-bit margin (bounds-checked build)

struct Bc {
    int* err;
    int64_t margin;
};
__device__ __forceinline__ Bc bc_open(int* err) {
    if constexpr (kBoundsCheck) {
        return {err, err ? (int64_t)*reinterpret_cast<const volatile long long*>(err + 2) : 0};
    } else {
        return {nullptr, 0};
    }
}
__device__ __forceinline__ bool bc_fail(const Bc& bc, int site) {
    if (bc.err) atomicCAS(bc.err, 0, kDevErrBounds + site);
    return false;
}
// [p, p + n) inside [base, base + extent - margin).
__device__ __forceinline__ bool bc_global(const Bc& bc, const void* p, int64_t n, const void* base,
                                          int64_t extent, int site) {
    if constexpr (!kBoundsCheck) {
        return true;
    } else {
        const int64_t off = reinterpret_cast<const char*>(p) - reinterpret_cast<const char*>(base);
        return (off >= 0 && n >= 0 && off + n <= extent - bc.margin) ? true : bc_fail(bc, site);
    }
}
// A global range an asynchronous copy reads (a bulk copy the kernel then
// waits for): false (skip the copy) only if it leaves the buffer itself; a
// range inside the buffer but within the margin of its end is recorded and
// still copied, so that no wait depends on the margin.
__device__ __forceinline__ bool bc_global_async(const Bc& bc, const void* p, int64_t n, const void* base,
                                                int64_t extent, int site) {
    if constexpr (!kBoundsCheck) {
        return true;
    } else {
        const int64_t off = reinterpret_cast<const char*>(p) - reinterpret_cast<const char*>(base);
        if (off < 0 || n < 0 || off + n > extent) return bc_fail(bc, site);
        if (off + n > extent - bc.margin) bc_fail(bc, site);
        return true;
    }
}
// A TMA box origin: its innermost coordinate x (elements of `elem` bytes)
// on the 16-byte grid (false: skip the copy), and the box [x, x + box_x) x
// rows [y, y + 1) inside the tensor's [0, dim_x) x [0, dim_y) (recorded only:
// the copy unit fills what lies outside).
__device__ __forceinline__ bool bc_tma(const Bc& bc, int64_t x, int elem, int64_t box_x, int64_t dim_x,
                                       int64_t y, int64_t dim_y, int site_align, int site_range) {
    if constexpr (!kBoundsCheck) {
        return true;
    } else {
        if ((x * elem) % 16 != 0) return bc_fail(bc, site_align);
        if (x < 0 || x + box_x > dim_x || y < 0 || y >= dim_y) bc_fail(bc, site_range);
        return true;
    }
}
// 0 <= i and i + n <= limit (offsets in shared memory, tensor coordinates).
__device__ __forceinline__ bool bc_range(const Bc& bc, int64_t i, int64_t n, int64_t limit, int site) {
    if constexpr (!kBoundsCheck) {
        return true;
    } else {
        return (i >= 0 && n >= 0 && i + n <= limit) ? true : bc_fail(bc, site);
    }
}
// Bytes of dynamic shared memory this CTA was launched with.
__device__ __forceinline__ uint32_t dyn_smem_bytes() {
    uint32_t v;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
    return v;
}
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s: waits for a copy to land
// Limits by what is awaited, so that the wait at the root of a stall runs out
// first and its code is the one recorded: a copy landing (W or code stage)
// 2 s, a hand-off from another role 4 s, the final drains and the split-K
// slices 6 s.
__host__ __device__ constexpr unsigned long long wait_limit_ns(int code) {
    return (code == kDevErrTimeoutW || code == kDevErrTimeoutQ || code == kDevErrTimeoutMmaStage) ? kWaitLimitNs
           : (code == kDevErrTimeoutDrain || code == kDevErrTimeoutRecv) ? 3 * kWaitLimitNs
                                                                          : 2 * kWaitLimitNs;
}

// ---------------------------------------------------------------------------
// Nibble decoders (prmt.b32: 8 source bytes {b,a}; selector nibble bits 0-2
// pick a byte, bit 3 replicates its sign -- kept clear here).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Look up the 8 nibbles of a qs word w through a 16-entry byte table T.
// t0 = [T(L0), T(H0), T(L1), T(H1)], t1 = [T(L2), T(H2), T(L3), T(H3)],
// where byte k of w is (Hk << 4) | Lk.
__device__ __forceinline__ void lut16(uint32_t w, const uint32_t T0, const uint32_t T1,
                                      const uint32_t T2, const uint32_t T3, uint32_t& t0,
                                      uint32_t& t1) {
    const uint32_t sel = w & 0x77777777u;
    const uint32_t pick = ((w >> 1) & 0x44444444u) | 0x32103210u;
    t0 = prmt(prmt(T0, T1, sel), prmt(T2, T3, sel), pick);
    const uint32_t sel_hi = sel >> 16;
    t1 = prmt(prmt(T0, T1, sel_hi), prmt(T2, T3, sel_hi), pick >> 16);
}

// qs word -> int8x4 nibble values of elements i..i+3 (low nibbles) and
// 16+i..16+i+3 (high nibbles), through format WT's table.
template <int WT = kWtIQ4XS>
__device__ __forceinline__ void decode_s8(uint32_t w, uint32_t& lo4, uint32_t& hi4) {
    using T = WTables<WT>;
    uint32_t t0, t1;
    lut16(w, T::S0, T::S1, T::S2, T::S3, t0, t1);
    lo4 = prmt(t0, t1, 0x6420u);
    hi4 = prmt(t0, t1, 0x7531u);
}

// qs word (bytes k = 0..3 of sub-block element i = i0 + k) -> four fp16x2
// words (value[L_k], value[H_k]): the K-permuted order (element i, 16+i).
template <int WT = kWtIQ4XS>
__device__ __forceinline__ void decode_f16x2(uint32_t w, uint32_t out[4]) {
    using T = WTables<WT>;
    uint32_t t0, t1;
    lut16(w, T::U0, T::U1, T::U2, T::U3, t0, t1);
    const uint32_t h[4] = {prmt(t0, kF16HiByte, 0x4140u), prmt(t0, kF16HiByte, 0x4342u),
                           prmt(t1, kF16HiByte, 0x4140u), prmt(t1, kF16HiByte, 0x4342u)};
    const uint32_t off_bits = kF16Offset2;
    const __half2 off = *reinterpret_cast<const __half2*>(&off_bits);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h[k]), off);
        out[k] = *reinterpret_cast<uint32_t*>(&v);
    }
}

// Nibble c (0..15) of format WT as its integer value.
template <int WT = kWtIQ4XS>
__device__ __forceinline__ int wt_nibble_value(int c) {
    using T = WTables<WT>;
    const uint32_t word = (c < 4) ? T::S0 : (c < 8) ? T::S1 : (c < 12) ? T::S2 : T::S3;
    return (int)(int8_t)(uint8_t)(word >> (8 * (c & 3)));
}
// Byte-table entry for a qs byte j (low nibble L = element i, high nibble
// H = element 16+i): the fp16x2 word (value[L], value[H]) that decode_f16x2
// produces for that byte, exact (|value| <= 128).
template <int WT = kWtIQ4XS>
__device__ __forceinline__ uint32_t f16x2_byte_entry(int j) {
    const uint32_t lo = __half_as_ushort(__int2half_rn(wt_nibble_value<WT>(j & 15)));
    const uint32_t hi = __half_as_ushort(__int2half_rn(wt_nibble_value<WT>(j >> 4)));
    return lo | (hi << 16);
}
__device__ __forceinline__ void sts_u128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
// As lds_u32, but ordered after earlier barrier waits (for data that a copy
// or another warp writes while this kernel runs; lds_u32 is only for data
// fixed since the block-wide barrier of set-up).
__device__ __forceinline__ uint32_t lds_u32_ordered(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// 6-bit scale of sub-block j from the 8-byte header word pair
// hdr0 = d | scales_h << 16, hdr1 = scales_l[0..3].
__device__ __forceinline__ int iq4xs_ls(uint32_t hdr0, uint32_t hdr1, int j) {
    const int lo = (hdr1 >> (4 * j)) & 0xF;  // byte j/2, nibble j&1 == bits 4j..4j+3
    const int hi = (hdr0 >> (16 + 2 * j)) & 3;
    return lo | (hi << 4);
}
__device__ __forceinline__ float iq4xs_scale(uint32_t hdr0, uint32_t hdr1, int j) {
    const float d = __half2float(__ushort_as_half((unsigned short)(hdr0 & 0xFFFF)));
    return d * (float)(iq4xs_ls(hdr0, hdr1, j) - 32);
}

// One 18-byte block from the five 4-byte words starting at the block's
// address rounded down to 4 (raw[0..4]); `odd` = the block starts 2 bytes
// past that boundary.  Out: float(d) and the four words of nibbles.
__device__ __forceinline__ float b18_unpack(const uint32_t raw[5], bool odd, uint32_t q[4]) {
    const uint32_t sh = odd ? 16u : 0u;
    const uint32_t d16 = __funnelshift_rc(raw[0], raw[1], sh) & 0xFFFFu;
#pragma unroll
    for (int k = 0; k < 4; ++k) q[k] = __funnelshift_rc(raw[k], raw[k + 1], 16u + sh);
    return __half2float(__ushort_as_half((unsigned short)d16));
}

// Sub-block s (32 weights) of a weight row in format WT, loaded from global
// memory into six raw words (all loads in flight before any use), then
// unpacked into its fp32 scale and its four words of nibbles.
template <int WT>
__device__ __forceinline__ void wt_load_sub(const uint8_t* row, int64_t s, uint32_t raw[6]) {
    if constexpr (WT == kWtIQ4XS) {
        const uint8_t* blk = row + (s / kSubPerBlock) * kBlockBytes;
        const int j = (int)(s % kSubPerBlock);
        const uint2 hdr = __ldg(reinterpret_cast<const uint2*>(blk));
        const uint2 q01 = __ldg(reinterpret_cast<const uint2*>(blk + 8 + 16 * j));
        const uint2 q23 = __ldg(reinterpret_cast<const uint2*>(blk + 16 + 16 * j));
        raw[0] = hdr.x; raw[1] = hdr.y; raw[2] = q01.x; raw[3] = q01.y; raw[4] = q23.x; raw[5] = q23.y;
    } else {
        // block s at 18*s; its 4-byte-aligned start is 18*s - 2*(s & 1).  The
        // five words end at most 2 bytes past the block, inside the next
        // block of the row (the row's last block, s odd, ends exactly).
        const uint32_t* a = reinterpret_cast<const uint32_t*>(row + kB18Bytes * s - 2 * (s & 1));
#pragma unroll
        for (int k = 0; k < 5; ++k) raw[k] = __ldg(a + k);
        raw[5] = 0;
    }
}
// Bounds-checked build: the bytes wt_load_sub reads for sub-block s of
// `row` lie inside the weight buffer [base, base + extent).
template <int WT>
__device__ __forceinline__ bool wt_sub_in_bounds(const Bc& bc, const uint8_t* row, int64_t s,
                                                 const void* base, int64_t extent, int site) {
    if constexpr (WT == kWtIQ4XS) {
        const uint8_t* blk = row + (s / kSubPerBlock) * kBlockBytes;
        const int j = (int)(s % kSubPerBlock);
        return bc_global(bc, blk, 8, base, extent, site) &&
               bc_global(bc, blk + 8 + 16 * j, 16, base, extent, site);
    } else {
        return bc_global(bc, row + kB18Bytes * s - 2 * (s & 1), 20, base, extent, site);
    }
}
template <int WT>
__device__ __forceinline__ float wt_unpack_sub(const uint32_t raw[6], int64_t s, uint32_t q[4]) {
    if constexpr (WT == kWtIQ4XS) {
#pragma unroll
        for (int k = 0; k < 4; ++k) q[k] = raw[2 + k];
        return iq4xs_scale(raw[0], raw[1], (int)(s % kSubPerBlock));
    } else {
        return b18_unpack(raw, (s & 1) != 0, q);
    }
}

// ---------------------------------------------------------------------------
// PTX wrappers: shared-memory addresses, mbarriers, bulk copies, tcgen05.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// try_wait that may suspend the thread (up to `ns` nanoseconds) until the
// phase completes, instead of returning at once: a waiting warp then takes
// no issue slots from the warps that do the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase with the given parity to complete.  Returns
// false (without waiting further) once the CTA's abort flag is set, or after
// wait_limit_ns(code), in which case it sets the abort flag and records
// `code` in the device error word unless an earlier code is there (the first
// wait to run out is the one reported).  The first probe returns at once;
// later ones suspend for up to 0.1 ms.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* err, int code) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(a, parity, 100000u)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > wait_limit_ns(code)) {
            *abort_flag = 1;
            atomicCAS(err, 0, code);
            return false;
        }
    }
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 2D tiled TMA load into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
// 3D tiled TMA load (coordinates x, y, z) into this CTA's shared memory,
// completing on `bar` (the experts of a grouped launch: z = expert).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, int x, int yc, int zc, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(yc), "r"(zc), "r"(smem_u32(bar))
        : "memory");
}
// Contiguous bulk copy global -> this CTA's shared memory (16-byte aligned
// addresses, size a multiple of 16), completing on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// Programmatic dependent launch.  wait: block until the preceding grid in
// the stream has completed and its writes are visible (a no-op when the
// launch had no programmatic dependency).  launch_dependents: allow the next
// grid in the stream to start launching (it still waits before touching
// anything this grid reads or writes).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Thread-block clusters: the cluster barrier, this CTA's rank, and bulk
// copies into another CTA's shared memory.
// Split phases of the cluster barrier: arrive without waiting (no ordering,
// or releasing this thread's earlier memory accesses), and the matching wait
// (acquire).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Bulk copy from this CTA's shared memory (src) to the same-offset address
// dst_local in CTA `rank` of the cluster, completing `bytes` on that CTA's
// mbarrier at offset bar_local (16-byte aligned addresses, size a multiple
// of 16).
__device__ __forceinline__ void bulk_copy_to_rank(uint32_t dst_local, uint32_t src, uint32_t bytes,
                                                  uint32_t bar_local, uint32_t rank) {
    uint32_t dst, bar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(dst) : "r"(dst_local), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(bar) : "r"(bar_local), "r"(rank));
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "r"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// tcgen05 (5th-generation tensor core, tensor memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16, issued by one thread.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16, A read from tensor memory
// (row i of A in lane i; column c holds K elements 2c (low half) and 2c+1).
__device__ __forceinline__ void tc_mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// One lane of the (converged) warp returns true.
__device__ __forceinline__ bool elect_one() {
    uint32_t p;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(p));
    return p != 0;
}
// Arrive on `bar` once every tcgen05 operation this thread issued so far is complete.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// TMEM -> registers with the wait fused into the same asm statement, so the
// destination registers are defined only once the asynchronous loads have
// completed (with a separate wait the compiler may read or move them early).
// `taddr` is lane << 16 | column; each helper reads consecutive columns.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld48_wait(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%48];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%49];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47])
        : "r"(taddr), "r"(taddr + 32u)
        : "memory");
}
__device__ __forceinline__ void tmem_ld64_wait(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr), "r"(taddr + 32u)
        : "memory");
}

// As above, plus k = 1 or 2 more columns (`saddr`: per-row scales) read under
// the same wait: `n` columns from `taddr` into r[0..n-1], k columns into sw.
__device__ __forceinline__ void tmem_ld16_s1_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%16}, [%18];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(sw[0])
        : "r"(taddr + 0u), "r"(saddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld32_s1_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%32}, [%34];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(sw[0])
        : "r"(taddr + 0u), "r"(saddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld48_s1_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%49];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%50];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%48}, [%51];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(sw[0])
        : "r"(taddr + 0u), "r"(taddr + 32u), "r"(saddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld64_s1_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%65];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%66];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%64}, [%67];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(sw[0])
        : "r"(taddr + 0u), "r"(taddr + 32u), "r"(saddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld16_s2_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%18];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%16,%17}, [%19];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(sw[0]), "=r"(sw[1])
        : "r"(taddr + 0u), "r"(saddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld32_s2_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%34];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%32,%33}, [%35];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(sw[0]), "=r"(sw[1])
        : "r"(taddr + 0u), "r"(saddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld48_s2_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%50];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%51];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%48,%49}, [%52];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(sw[0]), "=r"(sw[1])
        : "r"(taddr + 0u), "r"(taddr + 32u), "r"(saddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld64_s2_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%66];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%67];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%64,%65}, [%68];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(sw[0]), "=r"(sw[1])
        : "r"(taddr + 0u), "r"(taddr + 32u), "r"(saddr)
        : "memory");
}

// Generated load shapes for half-tile epilogue groups (24 = 16 + 8, 40 = 32 + 8, 56 = 32 + 16 + 8).
__device__ __forceinline__ void tmem_ld24_wait(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%24];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%25];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23])
        : "r"(taddr + 0u), "r"(taddr + 16u)
        : "memory");
}
__device__ __forceinline__ void tmem_ld24_s1_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%25];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%26];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%24}, [%27];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(sw[0])
        : "r"(taddr + 0u), "r"(taddr + 16u), "r"(saddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld24_s2_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%26];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%27];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%24,%25}, [%28];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(sw[0]), "=r"(sw[1])
        : "r"(taddr + 0u), "r"(taddr + 16u), "r"(saddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld40_wait(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%40];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%32,%33,%34,%35,%36,%37,%38,%39}, [%41];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39])
        : "r"(taddr + 0u), "r"(taddr + 32u)
        : "memory");
}
__device__ __forceinline__ void tmem_ld40_s1_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%41];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%32,%33,%34,%35,%36,%37,%38,%39}, [%42];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%40}, [%43];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(sw[0])
        : "r"(taddr + 0u), "r"(taddr + 32u), "r"(saddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld40_s2_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%42];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%32,%33,%34,%35,%36,%37,%38,%39}, [%43];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%40,%41}, [%44];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(sw[0]), "=r"(sw[1])
        : "r"(taddr + 0u), "r"(taddr + 32u), "r"(saddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld56_wait(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%56];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%57];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%48,%49,%50,%51,%52,%53,%54,%55}, [%58];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55])
        : "r"(taddr + 0u), "r"(taddr + 32u), "r"(taddr + 48u)
        : "memory");
}
__device__ __forceinline__ void tmem_ld56_s1_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%57];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%58];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%48,%49,%50,%51,%52,%53,%54,%55}, [%59];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%56}, [%60];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(sw[0])
        : "r"(taddr + 0u), "r"(taddr + 32u), "r"(taddr + 48u), "r"(saddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld56_s2_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%58];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%59];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%48,%49,%50,%51,%52,%53,%54,%55}, [%60];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%56,%57}, [%61];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(sw[0]), "=r"(sw[1])
        : "r"(taddr + 0u), "r"(taddr + 32u), "r"(taddr + 48u), "r"(saddr)
        : "memory");
}

// Load W consecutive accumulator columns (and SC scale columns) and wait.
template <int W, int SC>
__device__ __forceinline__ void tmem_ld_cols_wait(uint32_t taddr, uint32_t saddr, uint32_t* r,
                                                  uint32_t* sw) {
    static_assert(SC >= 0 && SC <= 2, "scale columns");
    if constexpr (W == 16) {
        if constexpr (SC == 0) tmem_ld16_wait(taddr, r);
        else if constexpr (SC == 1) tmem_ld16_s1_wait(taddr, saddr, r, sw);
        else tmem_ld16_s2_wait(taddr, saddr, r, sw);
    } else if constexpr (W == 24) {
        if constexpr (SC == 0) tmem_ld24_wait(taddr, r);
        else if constexpr (SC == 1) tmem_ld24_s1_wait(taddr, saddr, r, sw);
        else tmem_ld24_s2_wait(taddr, saddr, r, sw);
    } else if constexpr (W == 32) {
        if constexpr (SC == 0) tmem_ld32_wait(taddr, r);
        else if constexpr (SC == 1) tmem_ld32_s1_wait(taddr, saddr, r, sw);
        else tmem_ld32_s2_wait(taddr, saddr, r, sw);
    } else if constexpr (W == 40) {
        if constexpr (SC == 0) tmem_ld40_wait(taddr, r);
        else if constexpr (SC == 1) tmem_ld40_s1_wait(taddr, saddr, r, sw);
        else tmem_ld40_s2_wait(taddr, saddr, r, sw);
    } else {
        static_assert(W == 48, "supported widths: 16, 24, 32, 40, 48");
        if constexpr (SC == 0) tmem_ld48_wait(taddr, r);
        else if constexpr (SC == 1) tmem_ld48_s1_wait(taddr, saddr, r, sw);
        else tmem_ld48_s2_wait(taddr, saddr, r, sw);
    }
}

// Registers -> TMEM: 16 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
// Registers -> TMEM: one 32-bit column of this thread's lane.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
// Every tcgen05.st this thread issued has completed.
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major, no swizzle: core matrices of
// 8 rows x 16 bytes stored contiguously; `lbo` = byte distance between
// core matrices adjacent along K, `sbo` = along M/N.  Bits 46-48 = 0b001.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major,
// N = n (multiple of 16 for M = 128), M = 128.
__host__ __device__ constexpr uint32_t idesc_f16_m128(int n) {
    return (1u << 4)                        // D format: F32
           | (0u << 7) | (0u << 10)         // A, B format: F16
           | ((uint32_t)(n >> 3) << 17)     // N >> 3
           | ((uint32_t)(kTileN >> 4) << 24);  // M >> 4
}

// ---------------------------------------------------------------------------
// Host-side launchers (defined in the kernel translation units).
// ---------------------------------------------------------------------------
struct DevCtx;  // per-device state kept by api.cu

// tc_operand: NULL, or where to write the prepared tensor-core operand too.
// err: the device error word (kErrWords ints); kernels of the bounds-checked
// build record misses there.
cudaError_t launch_quantize_q8_1(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* qs,
                                 void* ds, void* tc_operand, int* err, cudaStream_t stream);
cudaError_t launch_dequantize(const void* w, int wt, int64_t N, int64_t K, void* out,
                              int out_dtype, int* err, cudaStream_t stream);
// num_sms picks the launch shape (grids of more than two CTAs per SM run
// with more resident CTAs).
cudaError_t launch_matmul_dp4a(const void* w, int wt, int64_t N, int64_t K, const int8_t* qs,
                               const void* ds, int64_t M, float* y, int64_t ldy, int* err,
                               int num_sms, cudaStream_t stream);
// G experts in one launch: expert g has W (format wt) at w + g *
// expert_stride and the Q8_1 / output rows [row_offsets[g], row_offsets[g+1])
// (device array).
cudaError_t launch_matmul_dp4a_grouped(const void* w, int wt, int64_t expert_stride, int64_t G, int64_t N,
                                       int64_t K, const int8_t* qs, const void* ds,
                                       const int32_t* row_offsets, int64_t total_rows, float* y,
                                       int64_t ldy, int* err, cudaStream_t stream);
// Programmatic dependent launch on (default) or off for every launch.
bool pdl_enabled();
// `encode` is the driver's cuTensorMapEncodeTiled; `err` the device error word.
// Activations: the Q8_1 arrays (qs 16-byte aligned: its rows are staged by
// TMA) when tc_operand is NULL, else the prepared operand alone (qs, ds
// unused).  skip_w_stage >= 0 leaves that W stage of every CTA unissued
// (tests of the bounded waits); -1 in every ordinary call.
// Warp-level MMA path (every weight format wt): activation tiles of
// mma_tile_rows(M) rows (8, 16, 24 or 32); K % 512 == 0; qs 16-byte aligned
// (staged by TMA), ds read directly.
int mma_tile_rows(int64_t M);
// The grouped (mixture-of-experts) form of the warp-MMA path: expert g's W
// (format wt) at w + g * expert_stride (a multiple of 16), its rows
// [row_offsets[g], row_offsets[g+1]) of qs / ds / y; K % 512 == 0.
cudaError_t launch_matmul_mma_grouped(const void* w, int wt, int64_t expert_stride, int64_t G, int64_t N,
                                      int64_t K, const int8_t* qs, const void* ds, const int32_t* row_offsets,
                                      int64_t total_rows, float* y, int64_t ldy, void* encode, int* err,
                                      int num_sms, int skip_w_stage, cudaStream_t stream);
// Grouped (mixture-of-experts) matmul on the tcgen05 kernel (Q8_1 form,
// IQ4_XS, K % 512 == 0): activation tiles of tc_mtile(mean rows per expert
// slot) rows, one CTA per (row tile, expert tile), no K split.
cudaError_t launch_matmul_tc_grouped(const void* w, int64_t expert_stride, int64_t G, int64_t N, int64_t K,
                                     const int8_t* qs, const void* ds, const int32_t* row_offsets,
                                     int64_t total_rows, float* y, int64_t ldy, void* encode, int* err,
                                     cudaStream_t stream);
// Test override of the warp-MMA launch: weight rows per CTA, K splits and
// CTAs per SM (1, 2); 0 = the launch model's choice.
void mma_force_config(int rows_per_cta, int k_splits, int ctas_per_sm);
// The warp-MMA launch the path takes for (M, N, K): weight rows per CTA, K
// splits (cluster size) and CTAs per SM (the launch model's choice, or the
// forced one).
void mma_launch_config(int64_t M, int64_t N, int64_t K, int num_sms, int* rows, int* splits, int* ctas_per_sm);
// Measured warp-MMA launches: count entries of 6 int64 (N, K, activation-tile
// rows 8/16/24/32, rows per CTA, K splits, CTAs per SM); 0 clears.  -1 on a
// value out of range (nothing installed).
int mma_set_launch_table(const int64_t* entries, int count);
cudaError_t launch_matmul_mma(const void* w, int wt, int64_t N, int64_t K, const int8_t* qs, const void* ds,
                              int64_t M, float* y, int64_t ldy, void* encode, int* err, int num_sms,
                              int skip_w_stage, cudaStream_t stream);
cudaError_t launch_matmul_tc(const void* w, int wt, int64_t N, int64_t K, const int8_t* qs,
                             const void* ds, const void* tc_operand, int64_t M, float* y,
                             int64_t ldy, void* encode, int* err, int num_sms, int skip_w_stage,
                             cudaStream_t stream);

}  // namespace iq4xs
