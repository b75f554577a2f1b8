// kda_internal.h -- declarations shared by the library's translation units.
//
// Data flow of one kda_fwd call (all on the caller's stream):
//   1. schedule kernel: cu_seqlens (or B x T) -> per-sequence chunk offsets and
//      a table of 64-token chunks (start token, valid length); validates
//      cu_seqlens on the device.
//   2. chunk kernel (kda_prep.cu), one CTA per (chunk, head), fully parallel:
//      gate, in-chunk decays, the intra-chunk score matrices on tcgen05, the
//      unit-lower-triangular inverse, and the WY factors W, U on tcgen05.  It
//      writes one fixed-size record per (chunk, head) whose operand tiles are
//      already in the tcgen05 shared-memory layouts the next kernel uses.
//   3. recurrence kernel, which keeps the fp32 state in TMEM, streams the
//      records with bulk copies and runs the sequential chunk-to-chunk update
//      and outputs on tcgen05: kda_recur.cu (one CTA per (sequence, head,
//      value slice), for few pairs) or kda_recur_t.cu (one CTA per (sequence,
//      head) with the state transposed, for many pairs).
// Other paths: kda_fused.cu runs steps 2 and 3 in one cooperative launch;
// kda_segmented.cu splits few long sequences into segments, finds each
// segment's state map with the recurrence kernel in map mode, scans the maps
// and runs step 3 over the segments; kda_decode.cu handles T = 1 without
// steps 1-3.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "kda.h"

namespace kda {

constexpr int kChunk = 64;  // tokens per chunk
constexpr int kDim = 128;   // K = V = 128

// Per-(chunk, head) record written by the chunk kernel (byte offsets), laid
// out so that the recurrence kernel copies it whole and uses its pieces as
// tcgen05 B operands in place:
//   WQ : [scale*Qhat ; W], 128 rows (0..63 the decayed queries, 64..127 the W
//        rows of the chunk's tokens) x 128 key channels; MN-major (rows
//        contiguous inside a core matrix), 8-row groups 2048 B apart, 8-channel
//        groups 128 B apart.  B operand of X^T = S^T . [Q ; W]^T (N = 128, K = 128).
//   KT, AQ, AQL : 256 rows x 64 tokens, K-major (tokens contiguous inside a
//        core matrix), 8-token groups 128 B apart, 8-row groups 1024 B apart:
//        rows 0..127 = Ktilde^T (key channels), 128..191 = scale*Aqk as bf16
//        hi, 192..255 = the bf16 lo remainder (lo = bf16(x - hi)).  B operand of
//        the state and output update Delta^T . [Ktilde | Aqk_hi^T | Aqk_lo^T]
//        (N = 256, K = 64).
//   UT : U^T, [128 value channels][64 tokens] bf16 row-major.
//   GAM: chunk-end decay exp(G_last) per key channel, fp32 [128].
constexpr uint32_t kRecWQ = 0;
constexpr uint32_t kRecKT = 32768;
constexpr uint32_t kRecAQ = 49152;    // hi
constexpr uint32_t kRecAQL = 57344;   // lo
constexpr uint32_t kRecOperands = 65536;
constexpr uint32_t kRecUT = 65536;
constexpr uint32_t kRecGam = 81920;
constexpr uint32_t kRecBytes = 82432;

struct ChunkInfo {
    int32_t tok0;  // first token (row of the [total_tokens, H, 128] tensors)
    int32_t len;   // valid tokens, 1..64
};

// Workspace carve-up (all offsets 256-byte aligned).
struct Workspace {
    int32_t* flags;       // [0] = 1 when the schedule is valid
    int32_t* chunk_off;   // [N + 1] chunk prefix offsets per sequence
    ChunkInfo* info;      // [max_chunks]
    uint8_t* records;     // [max_chunks][H][kRecBytes]
    int32_t* ready;       // [max_chunks][H] record-complete flags (fused launch only)
    // segmented path only (segs > 0; see kda_segmented.cu): each sequence's
    // chunks split into segs runs
    int segs;             // segments per sequence (0: no segment area)
    int32_t* seg_off;     // [N * segs + 1] chunk offsets of the segments
    float* seg_maps;      // [N * segs][H][2][128][128]: X (state reached from zero, [k][v]),
                          // then M^T (linear part of the segment's state map, [j][k])
    float* seg_start;     // [N * segs][H][128][128]: state entering each segment, [k][v]
};

struct Problem {
    const void* q;
    const void* k;
    const void* v;
    const void* g;
    const void* beta;
    float scale;
    void* out;
    const float* A_log;
    const float* dt_bias;
    float lower_bound;
    const void* h0;
    kda_dtype_t h0_dtype;
    void* hT;
    kda_dtype_t hT_dtype;
    const int32_t* cu;
    int32_t N;       // sequences
    int32_t B, T, H;
    int64_t total_tokens;
    int64_t max_chunks;
    bool qk_norm;    // scale every q and k row to unit L2 norm first (kda_fwd_ex flag)
};

// eps of the q/k normalisation: x / sqrt(|x|^2 + eps)
constexpr float kL2NormEps = 1e-6f;

size_t workspace_bytes(int64_t max_chunks, int64_t N, int64_t H, int segs);
Workspace carve_workspace(void* base, int64_t max_chunks, int64_t N, int64_t H, int segs);

// Error reporting (thread-local message).
kda_status_t set_error(kda_status_t s, const char* msg);
kda_status_t cuda_error(cudaError_t e, const char* where);
void clear_error();

// Library status word on the current device (see kda_device_status).
int* device_status_ptr();
constexpr int kStatusDeviceInput = 1;
constexpr int kStatusTimeout = 2;
constexpr int kStatusLayout = 4;  // a kernel found its shared-memory area misaligned (skipped its work)

// Kernel launchers (kda_prep.cu, kda_recur.cu, kda_recur_t.cu, kda_api.cu).
cudaError_t launch_schedule(const Problem& p, const Workspace& ws, int* status, cudaStream_t st);
cudaError_t launch_prep(const Problem& p, const Workspace& ws, int* status, cudaStream_t st);
// Single-token step (kda_decode.cu): T = 1 without cu_seqlens, no workspace.
bool decode_applies(const Problem& p);
cudaError_t launch_decode(const Problem& p, int* status, cudaStream_t st);

// Fused launch (kda_fused.cu): chunk kernel and transposed recurrence in one
// cooperative kernel.  fused_eligible says whether this device and problem
// can take it (forced: the caller asked for it explicitly).
bool fused_eligible(const Problem& p, bool forced);
cudaError_t launch_fused(const Problem& p, const Workspace& ws, int* status, cudaStream_t st);
inline size_t ready_bytes(int64_t max_chunks, int64_t H) {
    return (size_t)max_chunks * (size_t)H * sizeof(int32_t);
}

// recurrence: kind 0 = chosen from the problem shape, 1 = value-sliced, 2 = transposed;
// recur_choose resolves kind 0 to 1 or 2
int recur_choose(const Problem& p, int kind);
cudaError_t launch_recur(const Problem& p, const Workspace& ws, int* status, cudaStream_t st,
                         int kind);
// vs: value-slice width 32, 64 or 128 (0: chosen from the number of pairs)
cudaError_t launch_recur_sliced(const Problem& p, const Workspace& ws, int* status,
                                cudaStream_t st, int vs = 0);
// Segment maps (kda_recur.cu): for the N pseudo-sequences of p (the segments,
// ws.chunk_off = their chunk offsets) writes X and M^T into ws.seg_maps.
cudaError_t launch_recur_maps(const Problem& p, const Workspace& ws, int* status,
                              cudaStream_t st);

// Segmented path (kda_segmented.cu): split each sequence into segments, find
// each segment's affine state map, scan them, then run the recurrence on all
// segments at once.  segment_count gives the segments per sequence for the
// recurrence selection `kind` (0 automatic, 4 forced; 0 = path not taken).
int segment_count(int64_t N, int64_t H, int64_t max_chunks, int kind);
cudaError_t launch_seg_schedule(const Problem& p, const Workspace& ws, cudaStream_t st);
cudaError_t launch_seg_maps(const Problem& p, const Workspace& ws, int* status, cudaStream_t st);
cudaError_t launch_seg_scan(const Problem& p, const Workspace& ws, int* status, cudaStream_t st);
cudaError_t launch_seg_outputs(const Problem& p, const Workspace& ws, int* status,
                               cudaStream_t st);
cudaError_t launch_recur_transposed(const Problem& p, const Workspace& ws, int* status,
                                   cudaStream_t st);

kda_status_t selftest_tcgen05(const void* a, const void* b, float* d, int N, int K,
                              cudaStream_t stream);

}  // namespace kda
