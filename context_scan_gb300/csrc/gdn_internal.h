// gdn_internal.h -- launch interface shared by the host API and the kernels (not public).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kChunk = 64;
// packed-sequence pieces: ints per table entry (see ChainParams::piece_tab)
constexpr int kPieceFields = 8;
enum { PF_SEQ = 0, PF_CHUNK0, PF_NCHUNKS, PF_START, PF_END, PF_MS };

// WY tile pair of one chunk (tensor-core path): A diag(beta), then A diag(beta 2^Gx) (or
// 2^G for the decayed read). Each factor is lower triangular by 16 x 16 blocks and is stored,
// bf16, as the B operands of the four tcgen05 MMAs that multiply by it (one per 16 columns
// j): slab s holds rows 16 s .. 63 of columns 16 s .. 16 s + 15 as K-major 8 x 8 core matrices
// without swizzle (8 rows of 16 bytes each), row groups 128 bytes apart, its two 8-column
// halves wy_slab_lbo(s) bytes apart; the slabs follow one another from wy_slab0(s). No zeros
// above the diagonal blocks are stored, and MMA s covers rows 16 s .. 63 only (N = 64 - 16 s).
constexpr int kWyTileBytes = 5120;
constexpr int kWyPairBytes = 2 * kWyTileBytes;
__host__ __device__ constexpr int wy_slab0(int s) { return 128 * (18 * s - 2 * s * s); }
__host__ __device__ constexpr int wy_slab_lbo(int s) { return 128 * (8 - 2 * s); }
// byte offset of the 16-byte piece holding row `row`, columns 8 kg .. 8 kg + 7 of one factor
// (row >= 16 (kg / 2))
__host__ __device__ constexpr int wy_piece(int row, int kg) {
    return wy_slab0(kg >> 1) + (kg & 1) * wy_slab_lbo(kg >> 1) + ((row >> 3) - 2 * (kg >> 1)) * 128 +
           (row & 7) * 16;
}
static_assert(wy_slab0(4) == kWyTileBytes && wy_piece(63, 7) + 16 == kWyTileBytes &&
              wy_piece(16, 2) == wy_slab0(1), "WY tile format");

// Device error word, at the start of the caller's workspace. The first error a kernel
// records sticks (atomicCAS from 0); gdn_check_device_error reads and clears it.
struct DeviceError {
    unsigned code;    // 0 or a gdn_status value
    unsigned detail;  // which wait gave up (kernel-specific tag)
};

// One launch of the chain kernels: every (b, h, segment) is an independent "chain" that
// walks its segment's chunks in order, carrying the state on chip.
struct ChainParams {
    const void* q;
    const void* k;
    const void* v;
    const void* g;
    const void* beta;
    // Initial state of each chain: h_start + seg * h_start_seg_stride + (b*H + h)*K*V,
    // or zero when h_start == nullptr.
    const float* h_start;
    long long h_start_seg_stride;
    void* o;           // forward: [B,T,H,V] out dtype
    float* h_final;    // forward: written by chains whose segment is nseg_total-1 (nullable)
    float* M;          // summary: [nseg_total,B,H,K,K]
    float* S;          // summary: [nseg_total,B,H,K,V]
    // tcgen05 path: per-chunk WY factors, [B*H][T/64] pairs of kWyPairBytes (the format at
    // kWyTileBytes above); per-channel gates at bf16 inputs: [B*H][T/64][A diag(beta) | C],
    // fp32 64 x 64 row-major
    void* wy;
    int B, T, H, K, V;
    int seg_len;       // tokens per segment (multiple of 64)
    // tcgen05 path: chunks of segment 0 when it differs from the others (0 = the same):
    // segment s > 0 then starts at chunk first_chunks + (s - 1) * seg_len / 64
    int first_chunks;
    int seg_first;     // first segment this launch processes
    int nseg_run;      // segments this launch processes: seg_first .. seg_first+nseg_run-1
    int nseg_total;    // segments in the whole problem
    // forward: when non-null, the final state of segment s is also written to
    // h_out + (s + 1) * h_out_seg_stride + (b*H + h)*K*V (the state entering segment s + 1)
    float* h_out;
    long long h_out_seg_stride;
    // forward, tcgen05 path: when non-null, the state entering every chunk g (counted from
    // the start of the sequence) with g % seg_chunks == 0 that the chain walks is written to
    // H_seg + (g / seg_chunks)*B*H*K*V + (b*H + h)*K*V (the states entering the API's
    // segments when pieces and segments do not coincide)
    float* H_seg;
    int seg_chunks;
    // varlen (null otherwise): the batch is packed, sequence b holds tokens cu_seqlens[b] ..
    // cu_seqlens[b+1]-1 (B = number of sequences, T = total tokens, one segment); its chunks
    // are numbered from cu_chunks[b] (the last one may be partial) and the WY tiles are
    // [H][total_chunks], total_chunks = T/64 + B bounding the chunks of any split
    const int* cu_seqlens;
    const int* cu_chunks;
    int total_chunks;
    // packed sequences cut into pieces (tcgen05 path; null otherwise): chain (e, h) of this
    // launch runs entry e < *piece_n of piece_tab (B bounds the entries) -- kPieceFields ints:
    // sequence (-1: no chain), first chunk, chunks, start (-1: the sequence's h_start, else a slot of
    // piece_states), end (-1: the sequence's h_final, -2: not kept, else a slot), summary slot
    // (M, S at [slot][H][K][K|V]). Slots of piece_states are [slot][H][K][V] fp32.
    const int* piece_tab;
    const int* piece_n;
    float* piece_states;
    int in_bf16;
    int out_bf16;
    int decay_first;   // the read sees the decayed state (inclusive gate on the read side)
    int gate_k;        // g holds one gate per key channel, [B,T,H,K] (CUDA-core kernels only)
    // launch as the programmatic dependent of the preceding grid in the stream (the kernel
    // then finishes only after that grid has)
    int launch_dependent;
    // WY tiles of the fixed-length batch: only chunks wy_lo .. wy_lo + wy_cnt - 1 of every
    // (b, h) (wy_cnt = 0: wy_lo to the end)
    int wy_lo, wy_cnt;
    // WY tiles: when non-null, a grid of at most six CTAs per SM hands the chunks out one at
    // a time from this counter (zeroed before the launch); with launch_dependent it is
    // launched as the programmatic dependent of the preceding grid (and finishes only after
    // that grid has)
    unsigned* wy_queue;
    // WY tiles, one CTA per chunk: a counter the launch zeroes for a later queue launch
    unsigned* wy_queue_reset;
    DeviceError* err;
};

// fp32 CUDA-core kernels (any supported K/V, fp32 or bf16 inputs)
cudaError_t launch_simt_forward(const ChainParams& p, cudaStream_t s);
cudaError_t launch_simt_summary(const ChainParams& p, cudaStream_t s);
// per-channel gates (gate_k) with bf16 inputs: the chains by sub-block normalisation with their
// products on the warp-level tensor cores (routed from the two launchers above)
cudaError_t launch_kda_mma_chain(const ChainParams& p, bool summary, cudaStream_t s);
// ... whose per-chunk factors A diag(beta) and C ([chunk][2][64][64] fp32 at p.wy, chunks
// numbered as the WY tiles) this forms beforehand, one CTA per chunk
cudaError_t launch_kda_prep(const ChainParams& p, cudaStream_t s);
// In-order scan over consecutive pieces p_first .. P-1 of every (b, h): the state entering
// piece p_first is h_first ([BH][K][V], or zero when null); entering piece p+1 it is
// M[p] H + S[p] (M, S indexed by piece, [piece][BH][K][K|V]). The state entering every piece
// p > p_first is written to Hp[p] ([P][BH][K][V]) when Hp is non-null, and the state entering
// every piece p with p % nsub == 0 to H_seg[p / nsub] ([P/nsub][BH][K][V]) when H_seg is
// non-null; H_seg[0] is h_seg0 (or zero) when p_first > 0. With an error word (err non-null),
// K == V == 128 and at least one product to form, the products run on the tensor cores
// (launch_tc_scan), whose bounded waits report to err; otherwise on the CUDA cores.
cudaError_t launch_scan(const float* M, const float* S, const float* h_first, float* Hp,
                        float* H_seg, const float* h_seg0, int p_first, int P, int nsub, int BH,
                        int K, int V, cudaStream_t s, DeviceError* err = nullptr);
// the same scan on tcgen05 (gdn_scan_tc.cu), when tc_scan_supported
bool tc_scan_supported(const float* M, const float* S, int p_first, int P, int K, int V);
cudaError_t launch_tc_scan(const float* M, const float* S, const float* h_first, float* Hp,
                           float* H_seg, const float* h_seg0, int p_first, int P, int nsub, int BH,
                           DeviceError* err, cudaStream_t s);

// Packed sequences cut into pieces (gdn_varlen.cu): the plan's tables, in the workspace. tab1f
// [nseq] (piece 0 of every sequence, the first phase's forwards), tab1s [e_max] (the summaries
// of the middle pieces), tab2 [e_max] (the second phase's forwards), kPieceFields ints each;
// counts [8]: the entries of the three tables, the piece length chosen and the scan's jobs;
// seqinfo [4 nseq]: pieces, first state slot and first summary slot of each sequence
// ([nseq][3]), then the scan's jobs (the sequences cut into three pieces or more, in order).
struct PiecePlan {
    int* tab1f;
    int* tab1s;
    int* tab2;
    int* counts;
    int* seqinfo;
};
// whether any plan could cut a sequence (every sequence's chains in one wave, a sequence long
// enough for two pieces); when not, the chains run as before without the plan's launches
bool pieces_possible(int T, int nseq, int H, int sms);
// the scan over each job's piece summaries M, S ([slot][H][K][K|V], K = V = 128) into the state
// slots ([slot][H][K][V]) of its pieces 2 .. k-1, from the state entering piece 1, on at most
// `sms` CTAs; launched as the programmatic dependent of the summary grid before it (and the
// second phase as its own)
cudaError_t launch_piece_scan(const PiecePlan& pl, int nseq, int H, int e_max, int sms,
                              const float* M, const float* S, float* states, cudaStream_t s);

// varlen metadata: checks the caller's cu_seqlens [nseq+1] (0 first, T last, non-decreasing)
// and writes a checked copy to cu_out and cu_chunks[s] = sum over sequences before s of
// ceil(length / 64) (s = 0..nseq). A bad array is recorded in the error word
// (GDN_ERR_INVALID_ARG) and both outputs become all zeros (every sequence empty), so the
// kernels that read them stay inside the buffers.
cudaError_t launch_varlen_meta(const int* cu_in, int nseq, int T, int* cu_out, int* cu_chunks,
                               DeviceError* err, cudaStream_t s);
// the same check followed, in the same block, by the plan for the nseq sequences and H heads on
// `sms` SMs, with at most e_max pieces past the first ones (gdn_varlen.cu)
cudaError_t launch_varlen_meta_plan(const int* cu_in, int nseq, int T, int* cu_out, int* cu_chunks,
                                    DeviceError* err, int H, int sms, int e_max,
                                    const PiecePlan& pl, cudaStream_t s);

// State-gradient summaries (backward): chain (b, h, seg) walks segment seg's chunks from the
// last to the first, starting from dH_end[seg] ([nseg][B][H][K][V], or zero when null), and
// writes the gradient on the state entering the segment to dS[seg]. dO has the output dtype.
struct StateGradParams {
    const void* q;
    const void* k;
    const void* g;
    const void* beta;
    const void* dO;
    const float* dH_end;
    float* dS;
    // when non-null, the gradient on the state leaving every chunk c (counted over the whole
    // sequence) is written to D_chunks + c*B*H*K*V + (b*H + h)*K*V ([T/64][B][H][K][V])
    float* D_chunks;
    // bf16 inputs with K == V == 128: when non-null, the forward's per-chunk WY tiles
    // ([B*H][T/64] pairs in the format at kWyTileBytes), whose second factor replaces the
    // kernel's own inverse
    const void* wy;
    int B, T, H, K, V;
    int seg_len, nseg;
    int in_bf16, do_bf16, decay_first;
};
cudaError_t launch_state_grad(const StateGradParams& p, cudaStream_t s);
// columns of the state gradient one CTA of launch_state_grad owns (its grid is
// B*H*nseg*(V/tile) CTAs, one per SM)
constexpr int state_grad_tile(int in_bf16) { return in_bf16 ? 64 : 32; }

// Per-chunk gradients of the backward: every (b, h, chunk c) independently, from the chunk's
// q, k, v, g, beta, dO, the state entering it (Hc[c]) and the gradient on the state leaving it
// (Dc[c]), both [T/64][B][H][K][V] fp32: dq, dk [B,T,H,K], dv [B,T,H,V], dg, dbeta [B,T,H],
// all fp32.
struct ChunkGradParams {
    const void* q;
    const void* k;
    const void* v;
    const void* g;
    const void* beta;
    const void* dO;
    const float* Hc;
    const float* Dc;
    float* dq;
    float* dk;
    float* dv;
    float* dg;
    float* dbeta;
    int B, T, H, K, V;
    int in_bf16, do_bf16, decay_first;
};
cudaError_t launch_chunk_grad(const ChunkGradParams& p, cudaStream_t s);
// the same with the products on the warp-level tensor-core path (tf32 operands; bf16 inputs)
cudaError_t launch_chunk_grad_mma(const ChunkGradParams& p, cudaStream_t s);
// dH_in[s] = M[s]^T dH_in[s+1] + dS[s] for s = nseg-1 .. 0, dH_in[nseg] = dht (or zero)
cudaError_t launch_state_grad_scan(const float* M, const float* dS, const float* dht,
                                   float* dH_in, int nseg, int BH, int K, int V, cudaStream_t s);

// tcgen05 tensor-core kernels (bf16 inputs, K == V == 128)
bool tc_supported(const ChainParams& p);
bool tc_runtime_ok();   // the driver entry point that encodes tensor maps is available
// a bounded wait that runs out on purpose (see gdn_selftest_wait_timeout)
cudaError_t launch_wait_selftest(DeviceError* err, long long limit, unsigned tag, cudaStream_t s);
cudaError_t launch_tc_wy(const ChainParams& p, cudaStream_t s);   // see wy_lo, wy_cnt, wy_queue
cudaError_t launch_tc_forward(const ChainParams& p, cudaStream_t s);
cudaError_t launch_tc_summary(const ChainParams& p, cudaStream_t s);
// the first piece's forward (fwd) and the summaries beside it (sum) as one grid, whose CTAs let
// a programmatic dependent start at once
cudaError_t launch_tc_phase1(const ChainParams& fwd, const ChainParams& sum, cudaStream_t s);

}  // namespace gdn
