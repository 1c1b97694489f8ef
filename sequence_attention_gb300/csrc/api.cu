// Host side of libditsp: status strings, the thread-local error message, the
// library's device status word, and the rank-partition bookkeeping
// (edge-dit.cpp "Parallel execution": SPSequenceSplit / SPAllToAll4DLayout;
// cache-dit "Context Parallelism": UAA uneven lengths, Any Head Num padding).
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "common.cuh"

namespace ditsp {

static thread_local char g_msg[512] = "no error";

dit_status fail(dit_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

dit_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(DIT_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    return DIT_OK;
}

// Status word for calls made without their own d_status.  One per device
// that loads the module; its address is looked up per device on first use.
__device__ int g_device_status;

static constexpr int kMaxDevices = 64;
static std::atomic<int*> g_status_addr[kMaxDevices];
static std::atomic<int> g_sms[kMaxDevices];

int* default_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int* p = g_status_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_device_status) != cudaSuccess) return nullptr;
        p = static_cast<int*>(a);
        g_status_addr[dev].store(p, std::memory_order_release);
    }
    return p;
}

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int n = g_sms[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        g_sms[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace ditsp

using namespace ditsp;

extern "C" const char* dit_status_string(dit_status s) {
    switch (s) {
        case DIT_OK: return "DIT_OK";
        case DIT_ERR_INVALID_ARG: return "DIT_ERR_INVALID_ARG";
        case DIT_ERR_UNSUPPORTED: return "DIT_ERR_UNSUPPORTED";
        case DIT_ERR_CUDA: return "DIT_ERR_CUDA";
        case DIT_ERR_TIMEOUT: return "DIT_ERR_TIMEOUT";
        case DIT_ERR_RANGE: return "DIT_ERR_RANGE";
    }
    return "DIT_ERR_UNKNOWN";
}

extern "C" const char* dit_last_error(void) { return g_msg; }

extern "C" dit_status dit_device_status(int* out_code, int reset) {
    NvtxRange nvtx_range("dit_device_status");
    if (!out_code) return fail(DIT_ERR_INVALID_ARG, "dit_device_status: out_code is NULL");
    int* p = default_status_word();
    if (!p) return fail(DIT_ERR_CUDA, "dit_device_status: no device status word");
    int v = 0;
    cudaError_t e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "dit_device_status: %s", cudaGetErrorString(e));
    if (reset) {
        int z = 0;
        e = cudaMemcpy(p, &z, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "dit_device_status: %s", cudaGetErrorString(e));
    }
    *out_code = v;
    return DIT_OK;
}

// Balanced split: of n parts, the first S mod n get one extra row.
static void split(int S, int n, int* len, int* off, int base) {
    int q = S / n, extra = S % n, acc = base;
    for (int i = 0; i < n; ++i) {
        len[i] = q + (i < extra ? 1 : 0);
        off[i] = acc;
        acc += len[i];
    }
}

extern "C" dit_status dit_sp_layout_init_ex(int B, int S, int H, int D, int U, int R, int flags,
                                            dit_sp_layout* out) {
    NvtxRange nvtx_range("dit_sp_layout_init_ex");
    if (!out) return fail(DIT_ERR_INVALID_ARG, "dit_sp_layout_init: out is NULL");
    if (B < 1 || H < 1 || D < 1 || S < 0)
        return fail(DIT_ERR_INVALID_ARG, "dit_sp_layout_init: need B,H,D >= 1 and S >= 0");
    if (U < 1 || U > DIT_MAX_U || R < 1 || R > DIT_MAX_R || U * R > DIT_MAX_RANKS)
        return fail(DIT_ERR_INVALID_ARG,
                    "dit_sp_layout_init: need 1<=U<=%d, 1<=R<=%d, U*R<=%d (got U=%d R=%d)",
                    DIT_MAX_U, DIT_MAX_R, DIT_MAX_RANKS, U, R);
    if (flags & ~(DIT_LAYOUT_NOPAD_HEADS | DIT_LAYOUT_PAD_LCM64))
        return fail(DIT_ERR_INVALID_ARG, "dit_sp_layout_init: unknown flags 0x%x", flags);
    long long S_pad = S;
    if (flags & DIT_LAYOUT_PAD_LCM64) {
        long long a = U * R, b = 64;             // lcm(U*R, 64)
        while (b) { const long long t = a % b; a = b; b = t; }
        const long long m = (long long)U * R * 64 / a;
        S_pad = (S + m - 1) / m * m;
    }
    const bool nopad = (flags & DIT_LAYOUT_NOPAD_HEADS) != 0;
    const int Hl = (H + U - 1) / U;
    const long long Hp = nopad ? H : (long long)Hl * U;
    // every buffer of the path must be indexable with int64 and its row
    // count with int32
    const double elems = 3.0 * B * (double)S_pad * (double)Hp * D;
    if (elems > 4.0e18 || (double)Hp * D > 2.0e9 || S_pad > 2000000000LL)
        return fail(DIT_ERR_INVALID_ARG, "dit_sp_layout_init: sizes overflow");
    memset(out, 0, sizeof(*out));
    out->B = B; out->S = S; out->H = H; out->D = D; out->U = U; out->R = R;
    out->Hp = (int)Hp; out->Hl = Hl;
    out->S_pad = (int)S_pad;
    out->flags = flags;
    if (nopad) {
        split(H, U, out->head_len, out->head_off, 0);
    } else {
        for (int v = 0; v < U; ++v) {
            out->head_len[v] = Hl;
            out->head_off[v] = v * Hl;
        }
    }
    split((int)S_pad, R, out->ring_len, out->ring_off, 0);
    int cap = 0;
    for (int r = 0; r < R; ++r) {
        if (out->ring_len[r] > cap) cap = out->ring_len[r];
        split(out->ring_len[r], U, out->rank_len + r * U, out->rank_off + r * U, out->ring_off[r]);
    }
    out->S_cap = cap;
    for (int r = 0; r < R; ++r) {
        const int real = S - out->ring_off[r];
        out->ring_real[r] = real < 0 ? 0 : (real > out->ring_len[r] ? out->ring_len[r] : real);
    }
    return DIT_OK;
}

extern "C" dit_status dit_sp_layout_init(int B, int S, int H, int D, int U, int R, dit_sp_layout* out) {
    NvtxRange nvtx_range("dit_sp_layout_init");
    return dit_sp_layout_init_ex(B, S, H, D, U, R, 0, out);
}

extern "C" dit_status dit_sp_a2a_counts(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes,
                                        int rank, int64_t* sc, int64_t* sd, int64_t* rc,
                                        int64_t* rd) {
    NvtxRange nvtx_range("dit_sp_a2a_counts");
    if (!L || !sc || !sd || !rc || !rd)
        return fail(DIT_ERR_INVALID_ARG, "dit_sp_a2a_counts: NULL argument");
    if (nplanes < 1 || nplanes > 3 || rank < 0 || rank >= L->U * L->R)
        return fail(DIT_ERR_INVALID_ARG, "dit_sp_a2a_counts: bad nplanes or rank");
    if (dir != DIT_SEQ_TO_HEAD && dir != DIT_HEAD_TO_SEQ)
        return fail(DIT_ERR_INVALID_ARG, "dit_sp_a2a_counts: bad direction");
    const int U = L->U, r = rank / U, me = rank - r * U;
    const int64_t row = (int64_t)nplanes * L->B * L->D;     // elements per row and head
    int64_t sacc = 0, racc = 0;
    for (int p = 0; p < U; ++p) {
        const int64_t rows_p = L->rank_len[r * U + p], rows_me = L->rank_len[rank];
        const int64_t heads_p = L->head_len[p], heads_me = L->head_len[me];
        // seq->head: I send my rows of p's heads and get p's rows of mine;
        // head->seq: I send p its rows of my heads and get my rows of p's
        sc[p] = row * (dir == DIT_SEQ_TO_HEAD ? rows_me * heads_p : rows_p * heads_me);
        rc[p] = row * (dir == DIT_SEQ_TO_HEAD ? rows_p * heads_me : rows_me * heads_p);
        sd[p] = sacc; sacc += sc[p];
        rd[p] = racc; racc += rc[p];
    }
    return DIT_OK;
}
