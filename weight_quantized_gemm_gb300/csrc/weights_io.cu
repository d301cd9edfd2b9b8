// Packed-weight files: qgemm_save / qgemm_load_info / qgemm_load (include/qgemm.h).
//
// A file holds one packed layer, so that a model's weights are quantized once and loaded ready
// to run: a 64-byte little-endian header, then the packed weights Bp, then the {offset, scale}
// table T (absent in FLOAT mode), both exactly as qgemm_pack writes them.
//   offset  0  char[8]  magic "QGEMMW\0\1"
//           8  u32      format version (1)
//          12  u32      header bytes (64)
//          16  i32 x 5  K, N, mode, block (as given to qgemm_pack, 0 = per channel), w_dtype
//          36  u32      CRC-32 of the payload (Bp then T)
//          40  u64      Bp bytes
//          48  u64      T bytes
//          56  u64      0 (reserved)
// The checksum is the common reflected CRC-32 (polynomial 0xEDB88320, initial value and final
// XOR 0xFFFFFFFF), computed with a 256-entry table.
#include <stdio.h>
#include <string.h>

#include <new>
#include <vector>

#include "../../include/qgemm.h"
#include "internal.h"

namespace {

constexpr char kMagic[8] = {'Q', 'G', 'E', 'M', 'M', 'W', '\0', '\1'};
constexpr uint32_t kVersion = 1;
constexpr uint32_t kHeaderBytes = 64;
constexpr size_t kChunk = size_t(8) << 20;   // file and staging transfers in 8 MiB pieces

struct Crc32 {
    uint32_t table[256];
    Crc32() {
        for (uint32_t i = 0; i < 256; ++i) {
            uint32_t c = i;
            for (int k = 0; k < 8; ++k) c = (c & 1u) ? (0xEDB88320u ^ (c >> 1)) : (c >> 1);
            table[i] = c;
        }
    }
    // Continues a running CRC (start from 0) over n more bytes.
    uint32_t update(uint32_t crc, const uint8_t* p, size_t n) const {
        uint32_t c = crc ^ 0xFFFFFFFFu;
        for (size_t i = 0; i < n; ++i) c = table[(c ^ p[i]) & 0xFFu] ^ (c >> 8);
        return c ^ 0xFFFFFFFFu;
    }
};
const Crc32& crc32() {
    static const Crc32 c;
    return c;
}

void put32(uint8_t* p, uint32_t v) {
    for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
void put64(uint8_t* p, uint64_t v) {
    for (int i = 0; i < 8; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
uint32_t get32(const uint8_t* p) {
    uint32_t v = 0;
    for (int i = 0; i < 4; ++i) v |= (uint32_t)p[i] << (8 * i);
    return v;
}
uint64_t get64(const uint8_t* p) {
    uint64_t v = 0;
    for (int i = 0; i < 8; ++i) v |= (uint64_t)p[i] << (8 * i);
    return v;
}

struct Header {
    int K, N, mode, block, w_dtype;
    uint32_t crc;
    uint64_t bp_bytes, t_bytes;
};

struct File {
    FILE* f = nullptr;
    ~File() {
        if (f) fclose(f);
    }
};

// Reads and checks the header; the sizes must be the ones the shape implies.
int read_header(FILE* f, const char* path, Header* h) {
    uint8_t b[kHeaderBytes];
    if (fread(b, 1, kHeaderBytes, f) != kHeaderBytes) return qg::api_fail(QGEMM_ERR_IO, "short weight-file header");
    if (memcmp(b, kMagic, 8) != 0) return qg::api_fail(QGEMM_ERR_IO, "not a packed-weight file (bad magic)");
    if (get32(b + 8) != kVersion || get32(b + 12) != kHeaderBytes)
        return qg::api_fail(QGEMM_ERR_IO, "unsupported packed-weight file version");
    h->K = (int)get32(b + 16);
    h->N = (int)get32(b + 20);
    h->mode = (int)get32(b + 24);
    h->block = (int)get32(b + 28);
    h->w_dtype = (int)get32(b + 32);
    h->crc = get32(b + 36);
    h->bp_bytes = get64(b + 40);
    h->t_bytes = get64(b + 48);
    size_t tb = 0;
    const size_t pb = qg::api_packed_bytes(h->K, h->N, h->mode, h->block, h->w_dtype, &tb);
    if (h->N < 1 || pb == 0 || pb != h->bp_bytes || tb != h->t_bytes)
        return qg::api_fail(QGEMM_ERR_IO, "weight-file header is inconsistent with its shape");
    (void)path;
    return QGEMM_OK;
}

// Copies n bytes between host memory and (on_device) device memory, or host to host.
int copy_out(void* dst, const uint8_t* src, size_t n, int on_device, cudaStream_t s) {
    if (!on_device) {
        memcpy(dst, src, n);
        return QGEMM_OK;
    }
    cudaError_t e = cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return qg::api_fail(QGEMM_ERR_CUDA, cudaGetErrorString(e));
    return QGEMM_OK;
}
int copy_in(uint8_t* dst, const void* src, size_t n, int on_device, cudaStream_t s) {
    if (!on_device) {
        memcpy(dst, src, n);
        return QGEMM_OK;
    }
    cudaError_t e = cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return qg::api_fail(QGEMM_ERR_CUDA, cudaGetErrorString(e));
    return QGEMM_OK;
}

}  // namespace

extern "C" {

int qgemm_save(const char* path, int K, int N, int mode, int block, int w_dtype, const void* Bp, const float* T,
               int on_device, void* stream) {
    if (!path || (on_device != 0 && on_device != 1)) return qg::api_fail(QGEMM_ERR_ARG, "null path or bad on_device");
    size_t tb = 0;
    const size_t pb = qg::api_packed_bytes(K, N, mode, block, w_dtype, &tb);
    if (pb == 0 || N < 1) return qg::api_fail(QGEMM_ERR_ARG, "invalid packed-weight shape");
    if (!Bp || (tb && !T)) return qg::api_fail(QGEMM_ERR_ARG, "null Bp or T");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the payload's checksum first (one pass through a host staging buffer), then the file
    const Crc32& crc = crc32();
    std::vector<uint8_t> buf(kChunk);
    uint32_t c = 0;
    const struct {
        const void* p;
        size_t n;
    } parts[2] = {{Bp, pb}, {T, tb}};
    for (const auto& part : parts)
        for (size_t o = 0; o < part.n; o += kChunk) {
            const size_t n = part.n - o < kChunk ? part.n - o : kChunk;
            const int rc = copy_in(buf.data(), static_cast<const uint8_t*>(part.p) + o, n, on_device, s);
            if (rc != QGEMM_OK) return rc;
            c = crc.update(c, buf.data(), n);
        }
    uint8_t h[kHeaderBytes] = {};
    memcpy(h, kMagic, 8);
    put32(h + 8, kVersion);
    put32(h + 12, kHeaderBytes);
    put32(h + 16, (uint32_t)K);
    put32(h + 20, (uint32_t)N);
    put32(h + 24, (uint32_t)mode);
    put32(h + 28, (uint32_t)block);
    put32(h + 32, (uint32_t)w_dtype);
    put32(h + 36, c);
    put64(h + 40, pb);
    put64(h + 48, tb);
    File f;
    f.f = fopen(path, "wb");
    if (!f.f) return qg::api_fail(QGEMM_ERR_IO, "cannot open the weight file for writing");
    if (fwrite(h, 1, kHeaderBytes, f.f) != kHeaderBytes) return qg::api_fail(QGEMM_ERR_IO, "write failed");
    for (const auto& part : parts)
        for (size_t o = 0; o < part.n; o += kChunk) {
            const size_t n = part.n - o < kChunk ? part.n - o : kChunk;
            const int rc = copy_in(buf.data(), static_cast<const uint8_t*>(part.p) + o, n, on_device, s);
            if (rc != QGEMM_OK) return rc;
            if (fwrite(buf.data(), 1, n, f.f) != n) return qg::api_fail(QGEMM_ERR_IO, "write failed");
        }
    if (fclose(f.f) != 0) {
        f.f = nullptr;
        return qg::api_fail(QGEMM_ERR_IO, "close failed");
    }
    f.f = nullptr;
    return QGEMM_OK;
}

int qgemm_load_info(const char* path, int* K, int* N, int* mode, int* block, int* w_dtype) {
    if (!path || !K || !N || !mode || !block || !w_dtype) return qg::api_fail(QGEMM_ERR_ARG, "null argument");
    File f;
    f.f = fopen(path, "rb");
    if (!f.f) return qg::api_fail(QGEMM_ERR_IO, "cannot open the weight file");
    Header h;
    const int rc = read_header(f.f, path, &h);
    if (rc != QGEMM_OK) return rc;
    *K = h.K;
    *N = h.N;
    *mode = h.mode;
    *block = h.block;
    *w_dtype = h.w_dtype;
    return QGEMM_OK;
}

int qgemm_load(const char* path, void* Bp, size_t Bp_bytes, float* T, size_t T_bytes, int on_device, void* stream) {
    if (!path || !Bp || (on_device != 0 && on_device != 1)) return qg::api_fail(QGEMM_ERR_ARG, "null argument");
    File f;
    f.f = fopen(path, "rb");
    if (!f.f) return qg::api_fail(QGEMM_ERR_IO, "cannot open the weight file");
    Header h;
    int rc = read_header(f.f, path, &h);
    if (rc != QGEMM_OK) return rc;
    if (Bp_bytes < h.bp_bytes || (h.t_bytes && (!T || T_bytes < h.t_bytes)))
        return qg::api_fail(QGEMM_ERR_ARG, "destination buffers are smaller than the file's Bp / T");
    // The payload is read once into host memory and its checksum verified there; only those
    // verified bytes are then copied to the destination, so a file that changes while it is read
    // cannot put unchecked data into Bp or T.
    const Crc32& crc = crc32();
    const uint64_t total = h.bp_bytes + h.t_bytes;
    std::vector<uint8_t> payload;
    try {
        payload.resize((size_t)total);
    } catch (const std::bad_alloc&) {
        return qg::api_fail(QGEMM_ERR_IO, "no host memory for the weight file's payload");
    }
    uint32_t c = 0;
    for (uint64_t o = 0; o < total; o += kChunk) {
        const size_t n = (size_t)(total - o < kChunk ? total - o : kChunk);
        if (fread(payload.data() + o, 1, n, f.f) != n) return qg::api_fail(QGEMM_ERR_IO, "weight file is truncated");
        c = crc.update(c, payload.data() + o, n);
    }
    uint8_t extra;
    if (fread(&extra, 1, 1, f.f) != 0) return qg::api_fail(QGEMM_ERR_IO, "weight file has trailing bytes");
    if (c != h.crc) return qg::api_fail(QGEMM_ERR_IO, "weight file checksum mismatch");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const struct {
        void* p;
        uint64_t off, n;
    } parts[2] = {{Bp, 0, h.bp_bytes}, {T, h.bp_bytes, h.t_bytes}};
    for (const auto& part : parts) {
        if (part.n == 0) continue;
        rc = copy_out(part.p, payload.data() + part.off, (size_t)part.n, on_device, s);
        if (rc != QGEMM_OK) return rc;
    }
    return QGEMM_OK;
}

}  // extern "C"
