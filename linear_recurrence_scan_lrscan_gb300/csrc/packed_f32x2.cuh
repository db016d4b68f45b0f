// Packed fp32 pair arithmetic for the kernels whose per-element work is
// more than one fma (generated decays, complex maps).
#pragma once

namespace lrscan {

// Two fp32 lanes per instruction: the packed .f32x2 forms of PTX mul, fma
// and add (Blackwell).  Each half is rounded as the scalar instruction
// rounds it (round to nearest, subnormals kept), so the results are the
// scalar code's bit for bit.
__device__ __forceinline__ void mul_x2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "mul.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void add_x2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "add.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void fma_x2(float &d0, float &d1, float a0, float a1, float b0, float b1, float c0,
                                       float c1) {
    asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\tmov.b64 pc, {%6, %7};\n\t"
        "fma.rn.f32x2 pd, pa, pb, pc;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// Element-wise d = a * b, d = a + b and d = a * b + c over V lanes, two per
// packed instruction (an odd last lane takes the scalar form).  d may be one
// of the operands.
template <int V>
__device__ __forceinline__ void vmul(float (&d)[V], const float (&a)[V], const float (&b)[V]) {
#pragma unroll
    for (int v = 0; v + 1 < V; v += 2) mul_x2(d[v], d[v + 1], a[v], a[v + 1], b[v], b[v + 1]);
    if (V & 1) d[V - 1] = __fmul_rn(a[V - 1], b[V - 1]);
}
template <int V>
__device__ __forceinline__ void vadd(float (&d)[V], const float (&a)[V], const float (&b)[V]) {
#pragma unroll
    for (int v = 0; v + 1 < V; v += 2) add_x2(d[v], d[v + 1], a[v], a[v + 1], b[v], b[v + 1]);
    if (V & 1) d[V - 1] = __fadd_rn(a[V - 1], b[V - 1]);
}
template <int V>
__device__ __forceinline__ void vfma(float (&d)[V], const float (&a)[V], const float (&b)[V], const float (&c)[V]) {
#pragma unroll
    for (int v = 0; v + 1 < V; v += 2) fma_x2(d[v], d[v + 1], a[v], a[v + 1], b[v], b[v + 1], c[v], c[v + 1]);
    if (V & 1) d[V - 1] = __fmaf_rn(a[V - 1], b[V - 1], c[V - 1]);
}

}  // namespace lrscan
