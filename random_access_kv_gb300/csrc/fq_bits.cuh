// Device-side bit stream helpers for the fixed-address code layout [FibQuant §1, §2.3]:
// record m at stream bit m*R, indices LSB first, stream bit i = bit (i mod 32) of word i/32.
#pragma once

#include <stdint.h>

namespace fq {

// Writes one record starting at an arbitrary stream bit. Words wholly inside the record are
// stored plainly; a word shared with bits outside the record (another record, or bits beyond
// the call's range) is updated with two atomics that touch only this record's bits.
struct BitWriter {
    uint32_t *words;
    int64_t w;
    uint64_t acc;
    int n;
    uint32_t mask0;

    __device__ __forceinline__ BitWriter(uint32_t *codes, int64_t bitpos)
        : words(codes), w(bitpos >> 5), acc(0), n((int)(bitpos & 31)), mask0(~0u << (bitpos & 31)) {}

    __device__ __forceinline__ void emit(uint32_t val, uint32_t mask) {
        if (mask == 0xffffffffu) {
            words[w] = val;
        } else {
            atomicAnd(&words[w], ~mask);
            atomicOr(&words[w], val & mask);
        }
    }
    // Append the low B bits of v (B <= 16).
    __device__ __forceinline__ void put(uint32_t v, int B) {
        acc |= (uint64_t)v << n;
        n += B;
        if (n >= 32) {
            emit((uint32_t)acc, mask0);
            mask0 = ~0u;
            acc >>= 32;
            n -= 32;
            ++w;
        }
    }
    __device__ __forceinline__ void flush() {
        if (n > 0) emit((uint32_t)acc, mask0 & (0xffffffffu >> (32 - n)));
    }
};

// Reads consecutive B-bit fields starting at an arbitrary stream bit; loads a word only when
// the next field needs it, so it never reads past the record's last word.
struct BitReader {
    const uint32_t *words;
    int64_t w;
    uint64_t acc;
    int n;

    // With active = false nothing is read (and get() must not be called).
    __device__ __forceinline__ BitReader(const uint32_t *codes, int64_t bitpos, bool active = true)
        : words(codes), w((bitpos >> 5) + 1) {
        int off = (int)(bitpos & 31);
        acc = active ? (uint64_t)(__ldg(codes + (bitpos >> 5)) >> off) : 0ull;
        n = 32 - off;
    }
    __device__ __forceinline__ uint32_t get(int B) {
        if (n < B) {
            acc |= (uint64_t)__ldg(words + w) << n;
            ++w;
            n += 32;
        }
        uint32_t v = (uint32_t)acc & ((1u << B) - 1u);
        acc >>= B;
        n -= B;
        return v;
    }
};

}  // namespace fq
