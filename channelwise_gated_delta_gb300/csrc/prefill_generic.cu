// prefill_generic.cu -- chunkwise WY/UT prefill on CUDA cores, float32.
//
// Page "Reorder channelwise gated delta rule chunked hot loops for
// autovectorization" (pytorch/executorch PR #21021), second commit summary:
// for T != 1 the forward runs chunk by chunk, computing per-channel
// log-decay prefixes, causal query/key terms, a beta-folded triangular
// transform, WY pseudo-keys and pseudo-values, and the state carried from one
// chunk to the next; a ragged last chunk goes through the same code.
//
// The algebra (unrolling the per-token recurrence over one chunk of L tokens,
// local indices r, s; S0 = state at the chunk start; G = inclusive prefix sum
// of g over the chunk per key channel):
//   A[r,s] = beta_r sum_i k_ri k_si exp(G_ri - G_si)      s <  r  (else 0)
//   P[r,s] =        sum_i q_ri k_si exp(G_ri - G_si)      s <= r  (else 0)
//   Wk = (I + A)^-1 diag(beta) (exp(G) * K)    WY pseudo-keys    [L, dk]
//   Wv = (I + A)^-1 diag(beta) V               WY pseudo-values  [L, dv]
//   U  = Wv - Wk S0
//   O  = (exp(G) * Q) S0 + P U
//   S  = diag(exp(G_L)) S0 + (exp(G_L - G) * K)^T U
// Every exponent used is <= 0 (the decay between two tokens, taken in causal
// order), so nothing overflows whatever the strength of the decay.
//
// This is the general path: any supported (dk, dv, chunk) and both dtypes,
// float32 throughout, with exact pairwise decays.  Two kernels:
//   gdr_chunk_prep  one CTA per (batch, value head, chunk), all chunks in
//                   parallel: prefix sums, A and P, the unit-lower solve by
//                   forward substitution, and the per-chunk operands of the
//                   scan, written to the workspace;
//   gdr_chunk_scan  one CTA per (batch, value head, 32-column tile of dv),
//                   sequential over chunks: U, O and the state carry, with
//                   the state tile resident in shared memory.
#include "common.cuh"

namespace gdr {
namespace {

constexpr int kPrepThreads = 256;
constexpr int kScanThreads = 256;
constexpr int kScanBV = 32;

// Per (b, hv, chunk) workspace record, in floats:
//   Wk [C][dk] | Qt [C][dk] | Kh [C][dk] | Wv [C][dv] | P [C][C] | gam [dk]
struct ChunkLayout {
    int C, dk, dv;
    __host__ __device__ size_t wk() const { return 0; }
    __host__ __device__ size_t qt() const { return (size_t)C * dk; }
    __host__ __device__ size_t kh() const { return 2 * (size_t)C * dk; }
    __host__ __device__ size_t wv() const { return 3 * (size_t)C * dk; }
    __host__ __device__ size_t p() const { return 3 * (size_t)C * dk + (size_t)C * dv; }
    __host__ __device__ size_t gam() const { return p() + (size_t)C * C; }
    __host__ __device__ size_t floats() const {
        // keep each record a multiple of 4 floats (16 bytes)
        return (gam() + dk + 3) & ~(size_t)3;
    }
};

// TREE: the T <= C tokens of each (b, hv) are a draft-token tree given by
// parents[b][t] (-1 for a root, else an earlier token), solved as one chunk:
// prefix sums run along root paths and the ancestor relation replaces the
// causal order in A and P (page "Support TreeUpdateSolve kernel",
// trymirai/uzu PR #576).  No state carry is prepared.
template <typename Tin, bool TREE>
__global__ void __launch_bounds__(kPrepThreads)
    gdr_chunk_prep(const Tin *__restrict__ q, const Tin *__restrict__ k,
                   const Tin *__restrict__ v, const float *__restrict__ g,
                   const float *__restrict__ beta, float *__restrict__ ws,
                   const int2 *__restrict__ chunks, const int *__restrict__ parents, int T,
                   int HK, int HV, int dk, int dv, int C, int NC, int g_scalar) {
    extern __shared__ float smem[];
    const int ldk = dk + 1;  // padded rows: threads walking s hit distinct banks
    const int ldw = dk + dv;
    float *Ks = smem;               // [C][ldk]
    float *Qs = Ks + C * ldk;       // [C][ldk]
    float *Gs = Qs + C * ldk;       // [C][ldk]
    float *As = Gs + C * ldk;       // [C][C]
    float *Ws = As + C * C;         // [C][dk + dv]
    float *bs = Ws + C * ldw;       // [C]
    int *par = reinterpret_cast<int *>(bs + C);                          // [C] (TREE)
    unsigned long long *anc = reinterpret_cast<unsigned long long *>(
        reinterpret_cast<uintptr_t>(par + C + 1) & ~(uintptr_t)7);     // [C] (TREE)

    // The chunk: its first token row in the [rows][H][d] view of the inputs,
    // its length, and its record.  Dense batches: CTA (b, hv, c), record
    // (b, hv, c).  Packed variable-length batches: CTA (chunk, hv) over the
    // table of every sequence's chunks {first row, length}, record (chunk, hv).
    int hv, L;
    size_t tr0, rec_idx;
    if (chunks) {
        const int ci = blockIdx.x / HV;
        hv = blockIdx.x % HV;
        const int2 e = chunks[ci];
        tr0 = (size_t)e.x;
        L = e.y;
        rec_idx = (size_t)ci * HV + hv;
    } else {
        const int c = blockIdx.x % NC;
        const int head_idx = blockIdx.x / NC;
        hv = head_idx % HV;
        const int b = head_idx / HV;
        tr0 = (size_t)b * T + (size_t)c * C;
        L = min(C, T - c * C);
        rec_idx = (size_t)head_idx * NC + c;
    }
    const int hk = hv / (HV / HK);
    const int tid = threadIdx.x;
    const ChunkLayout lay{C, dk, dv};
    float *rec = ws + rec_idx * lay.floats();

    // Load the chunk (rows >= L are zero; a zero gate keeps G flat there).
    for (int idx = tid; idx < C * dk; idx += kPrepThreads) {
        const int r = idx / dk, i = idx % dk;
        float kv = 0.f, qv = 0.f, gv = 0.f;
        if (r < L) {
            const size_t tk = (tr0 + r) * HK + hk;
            kv = to_f32(k[tk * dk + i]);
            qv = to_f32(q[tk * dk + i]);
            // a scalar gate has one log-decay per token and head
            gv = g_scalar ? g[(tr0 + r) * HV + hv] : g[((tr0 + r) * HV + hv) * dk + i];
        }
        Ks[r * ldk + i] = kv;
        Qs[r * ldk + i] = qv;
        Gs[r * ldk + i] = gv;
    }
    for (int r = tid; r < C; r += kPrepThreads)
        bs[r] = r < L ? beta[(tr0 + r) * HV + hv] : 0.f;
    if (TREE) {
        const int b = blockIdx.x / NC / HV;
        for (int r = tid; r < C; r += kPrepThreads) par[r] = r < L ? parents[(size_t)b * T + r] : -1;
    }
    __syncthreads();

    if (TREE) {
        // Ancestor sets as bit masks (parents precede their children), and
        // the prefix sums of the log-decay along each token's root path.
        if (tid == 0) {
            for (int r = 0; r < C; ++r) {
                const int p = par[r];
                anc[r] = p < 0 ? 0ull : (anc[p] | (1ull << p));
            }
        }
        for (int i = tid; i < dk; i += kPrepThreads) {
            for (int r = 0; r < C; ++r) {
                const int p = par[r];
                Gs[r * ldk + i] += p < 0 ? 0.f : Gs[p * ldk + i];
            }
        }
    } else {
        // Per-channel inclusive prefix sum of the log-decay.
        for (int i = tid; i < dk; i += kPrepThreads) {
            float run = 0.f;
            for (int r = 0; r < C; ++r) {
                run += Gs[r * ldk + i];
                Gs[r * ldk + i] = run;
            }
        }
    }
    __syncthreads();

    // Causal key/key (A, beta-folded, strictly lower) and query/key (P) terms.
    float *Pg = rec + lay.p();
    for (int idx = tid; idx < C * C; idx += kPrepThreads) {
        const int r = idx / C, s = idx % C;
        // s is an earlier token r depends on: s <= r, or in a tree s == r or
        // an ancestor of r
        const bool below = TREE ? (s < r && ((anc[r] >> s) & 1ull)) : s < r;
        float a = 0.f, pp = 0.f;
        if ((below || s == r) && r < L) {
            const float *kr = Ks + r * ldk, *ks = Ks + s * ldk, *qr = Qs + r * ldk;
            const float *gr = Gs + r * ldk, *gs = Gs + s * ldk;
            for (int i = 0; i < dk; ++i) {
                const float e = expf(gr[i] - gs[i]);
                const float kse = ks[i] * e;
                a = fmaf(kr[i], kse, a);
                pp = fmaf(qr[i], kse, pp);
            }
        }
        As[r * C + s] = below ? bs[r] * a : 0.f;
        Pg[idx] = pp;
    }
    // Right-hand sides of the WY solve: diag(beta) [exp(G) * K | V].
    for (int idx = tid; idx < C * ldw; idx += kPrepThreads) {
        const int r = idx / ldw, col = idx % ldw;
        float x = 0.f;
        if (r < L) {
            if (col < dk) {
                x = bs[r] * Ks[r * ldk + col] * expf(Gs[r * ldk + col]);
            } else {
                const size_t tv = (tr0 + r) * HV + hv;
                x = bs[r] * to_f32(v[tv * dv + (col - dk)]);
            }
        }
        Ws[idx] = x;
    }
    __syncthreads();

    // (I + A) W = RHS by forward substitution; the columns are independent,
    // so each thread owns whole columns and walks the rows in order.
    for (int col = tid; col < ldw; col += kPrepThreads) {
        for (int r = 1; r < L; ++r) {
            float acc = Ws[r * ldw + col];
            const float *ar = As + r * C;
            for (int s = 0; s < r; ++s) acc = fmaf(-ar[s], Ws[s * ldw + col], acc);
            Ws[r * ldw + col] = acc;
        }
    }
    __syncthreads();

    // Scan operands: Wk, Wv, Qt = exp(G) Q, Kh = exp(G_L - G) K, gam = exp(G_L)
    // (a tree has no last token to carry the state to: no Kh, gam).
    const float *gl = Gs + (L - 1) * ldk;
    for (int idx = tid; idx < C * dk; idx += kPrepThreads) {
        const int r = idx / dk, i = idx % dk;
        const float gri = Gs[r * ldk + i];
        rec[lay.wk() + idx] = Ws[r * ldw + i];
        rec[lay.qt() + idx] = Qs[r * ldk + i] * expf(gri);
        if (!TREE) rec[lay.kh() + idx] = r < L ? Ks[r * ldk + i] * expf(gl[i] - gri) : 0.f;
    }
    for (int idx = tid; idx < C * dv; idx += kPrepThreads) {
        const int r = idx / dv, j = idx % dv;
        rec[lay.wv() + idx] = Ws[r * ldw + dk + j];
    }
    if (!TREE)
        for (int i = tid; i < dk; i += kPrepThreads) rec[lay.gam() + i] = expf(gl[i]);
}

// TREE: one chunk (the tree), outputs only: no state update, no ht.
template <typename Tin, bool TREE>
__global__ void __launch_bounds__(kScanThreads)
    gdr_chunk_scan(const float *__restrict__ ws, const float *h0, Tin *__restrict__ out,
                   float *ht, const int4 *__restrict__ seqs, int T_dense, int HV, int dk, int dv,
                   int C, int NC_dense) {
    extern __shared__ float smem[];
    const int ldk = dk + 1;
    const int ldc = C + 1;
    float *Ss = smem;                    // [dk][BV]   state tile
    float *Wk = Ss + dk * kScanBV;       // [C][ldk]
    float *Qt = Wk + C * ldk;            // [C][ldk]
    float *Kh = Qt + C * ldk;            // [C][ldk]
    float *Ps = Kh + C * ldk;            // [C][ldc]
    float *Us = Ps + C * ldc;            // [C][BV]
    float *Wv = Us + C * kScanBV;        // [C][BV]
    float *gam = Wv + C * kScanBV;       // [dk]

    const int ntile = dv / kScanBV;
    const int tile = blockIdx.x % ntile;
    const int hv = (blockIdx.x / ntile) % HV;
    const int b = blockIdx.x / ntile / HV;
    // The sequence: first token row, length, state slot, and where its chunk
    // records start and how far apart they are (dense: b's own rows, slot b,
    // records (b, hv, c); packed: {first row, length, slot, first chunk}
    // from the table, records (chunk, hv)).
    size_t tok0 = (size_t)b * T_dense, rec0 = ((size_t)b * HV + hv) * NC_dense, rec_step = 1;
    int T = T_dense, slot = b;
    if (seqs) {
        const int4 sd = seqs[b];
        tok0 = (size_t)sd.x;
        T = sd.y;
        slot = sd.z;
        rec0 = (size_t)sd.w * HV + hv;
        rec_step = HV;
    }
    const int NC = (T + C - 1) / C;
    const size_t head_idx = (size_t)slot * HV + hv;  // state slot
    const int j0 = tile * kScanBV;
    const int tid = threadIdx.x;
    const int jj = tid % kScanBV;        // column within the tile
    const int rr = tid / kScanBV;        // 0..7
    const ChunkLayout lay{C, dk, dv};

    for (int idx = tid; idx < dk * kScanBV; idx += kScanThreads) {
        const int i = idx / kScanBV, j = idx % kScanBV;
        Ss[idx] = h0 ? h0[(head_idx * dk + i) * dv + j0 + j] : 0.f;
    }

    for (int c = 0; c < NC; ++c) {
        const float *rec = ws + (rec0 + (size_t)c * rec_step) * lay.floats();
        const int t0 = c * C;
        const int L = min(C, T - t0);
        for (int idx = tid; idx < C * dk; idx += kScanThreads) {
            const int r = idx / dk, i = idx % dk;
            Wk[r * ldk + i] = rec[lay.wk() + idx];
            Qt[r * ldk + i] = rec[lay.qt() + idx];
            if (!TREE) Kh[r * ldk + i] = rec[lay.kh() + idx];
        }
        for (int idx = tid; idx < C * C; idx += kScanThreads)
            Ps[(idx / C) * ldc + idx % C] = rec[lay.p() + idx];
        for (int idx = tid; idx < C * kScanBV; idx += kScanThreads) {
            const int r = idx / kScanBV, j = idx % kScanBV;
            Wv[idx] = rec[lay.wv() + (size_t)r * dv + j0 + j];
        }
        if (!TREE)
            for (int i = tid; i < dk; i += kScanThreads) gam[i] = rec[lay.gam() + i];
        __syncthreads();

        // U = Wv - Wk S0
        for (int r = rr; r < C; r += kScanThreads / kScanBV) {
            float acc = Wv[r * kScanBV + jj];
            const float *w = Wk + r * ldk;
            for (int i = 0; i < dk; ++i) acc = fmaf(-w[i], Ss[i * kScanBV + jj], acc);
            Us[r * kScanBV + jj] = acc;
        }
        __syncthreads();

        // O = Qt S0 + P U
        for (int r = rr; r < L; r += kScanThreads / kScanBV) {
            float acc = 0.f;
            const float *qrow = Qt + r * ldk;
            for (int i = 0; i < dk; ++i) acc = fmaf(qrow[i], Ss[i * kScanBV + jj], acc);
            const float *prow = Ps + r * ldc;
            for (int s = 0; s <= r; ++s) acc = fmaf(prow[s], Us[s * kScanBV + jj], acc);
            out[((tok0 + t0 + r) * HV + hv) * dv + j0 + jj] = from_f32<Tin>(acc);
        }

        if (TREE) break;  // one chunk; no state to carry
        // S = diag(gam) S0 + Kh^T U   (new values kept in registers until
        // every thread is done reading S0)
        float snew[128 / (kScanThreads / kScanBV)];
        int n = 0;
        for (int i = rr; i < dk; i += kScanThreads / kScanBV, ++n) {
            float acc = gam[i] * Ss[i * kScanBV + jj];
            for (int r = 0; r < L; ++r) acc = fmaf(Kh[r * ldk + i], Us[r * kScanBV + jj], acc);
            snew[n] = acc;
        }
        __syncthreads();
        n = 0;
        for (int i = rr; i < dk; i += kScanThreads / kScanBV, ++n) Ss[i * kScanBV + jj] = snew[n];
        __syncthreads();
    }

    if (!TREE && ht) {
        for (int idx = tid; idx < dk * kScanBV; idx += kScanThreads) {
            const int i = idx / kScanBV, j = idx % kScanBV;
            ht[(head_idx * dk + i) * dv + j0 + j] = Ss[idx];
        }
    }
}

size_t prep_smem_bytes(int dk, int dv, int C) {
    // floats, then (trees) C parent indices and C 8-byte ancestor masks
    return sizeof(float) * ((size_t)3 * C * (dk + 1) + (size_t)C * C + (size_t)C * (dk + dv) + C) +
           sizeof(int) * (C + 2) + sizeof(unsigned long long) * C;
}
size_t scan_smem_bytes(int dk, int C) {
    return sizeof(float) * ((size_t)dk * kScanBV + (size_t)3 * C * (dk + 1) + (size_t)C * (C + 1) +
                            (size_t)2 * C * kScanBV + dk);
}

// Dense batches: chunks == seqs == nullptr, B x T from p.  Packed batches:
// nchunks chunk records and p.B sequence records.  Trees (TREE): p.T <=
// p.chunk tokens per batch element, parents [B][T] on the device.
template <typename Tin, bool TREE>
cudaError_t launch_generic_t(const Problem &p, void *workspace, const int2 *chunks, int nchunks,
                             const int4 *seqs, const int *parents, cudaStream_t stream) {
    const int C = p.chunk;
    const int NC = (p.T + C - 1) / C;
    float *ws = static_cast<float *>(workspace);
    const long long prep_blocks = chunks ? (long long)nchunks * p.HV : (long long)p.B * p.HV * NC;
    const long long scan_blocks = (long long)p.B * p.HV * (p.dv / kScanBV);
    if (prep_blocks > 0x7fffffffLL || scan_blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const size_t sp = prep_smem_bytes(p.dk, p.dv, C);
    const size_t ss = scan_smem_bytes(p.dk, C);
    cudaError_t e;
    e = cudaFuncSetAttribute(gdr_chunk_prep<Tin, TREE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sp);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gdr_chunk_scan<Tin, TREE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ss);
    if (e != cudaSuccess) return e;
    trace_begin(kKernChunkPrep, stream);
    gdr_chunk_prep<Tin, TREE><<<(unsigned)prep_blocks, kPrepThreads, sp, stream>>>(
        static_cast<const Tin *>(p.q), static_cast<const Tin *>(p.k),
        static_cast<const Tin *>(p.v), p.g, p.beta, ws, chunks, parents, p.T, p.HK, p.HV, p.dk,
        p.dv, C, NC, p.g_scalar);
    trace_end(kKernChunkPrep, stream);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    trace_begin(kKernChunkScan, stream);
    gdr_chunk_scan<Tin, TREE><<<(unsigned)scan_blocks, kScanThreads, ss, stream>>>(
        ws, p.h0, static_cast<Tin *>(p.out), p.ht, seqs, p.T, p.HV, p.dk, p.dv, C, NC);
    trace_end(kKernChunkScan, stream);
    return cudaGetLastError();
}

}  // namespace

size_t generic_prefill_workspace_bytes(const Problem &p) {
    const int NC = (p.T + p.chunk - 1) / p.chunk;
    const ChunkLayout lay{p.chunk, p.dk, p.dv};
    return sizeof(float) * lay.floats() * (size_t)p.B * p.HV * NC;
}

cudaError_t launch_generic_prefill(const Problem &p, void *workspace, cudaStream_t stream) {
    return p.bf16 ? launch_generic_t<__nv_bfloat16, false>(p, workspace, nullptr, 0, nullptr,
                                                           nullptr, stream)
                  : launch_generic_t<float, false>(p, workspace, nullptr, 0, nullptr, nullptr,
                                                   stream);
}

size_t generic_varlen_record_bytes(const Problem &p, long long nchunks) {
    const ChunkLayout lay{p.chunk, p.dk, p.dv};
    return sizeof(float) * lay.floats() * (size_t)nchunks * p.HV;
}

cudaError_t launch_generic_prefill_varlen(const Problem &p, void *records, const int2 *chunks,
                                          int nchunks, const int4 *seqs, cudaStream_t stream) {
    return p.bf16 ? launch_generic_t<__nv_bfloat16, false>(p, records, chunks, nchunks, seqs,
                                                           nullptr, stream)
                  : launch_generic_t<float, false>(p, records, chunks, nchunks, seqs, nullptr,
                                                   stream);
}

size_t generic_tree_record_bytes(const Problem &p) {
    const ChunkLayout lay{p.chunk, p.dk, p.dv};
    return sizeof(float) * lay.floats() * (size_t)p.B * p.HV;
}

cudaError_t launch_generic_tree(const Problem &p, void *records, const int *parents,
                                cudaStream_t stream) {
    return p.bf16 ? launch_generic_t<__nv_bfloat16, true>(p, records, nullptr, 0, nullptr,
                                                          parents, stream)
                  : launch_generic_t<float, true>(p, records, nullptr, 0, nullptr, parents,
                                                  stream);
}

}  // namespace gdr
