"""Writes tmem_ldst.inc: inline-PTX wrappers for the tcgen05.ld / tcgen05.st shapes
the kernels use. The operand lists are long (one register per 32-bit column), so
they are generated rather than typed.

Shapes (PTX ISA, tcgen05 "Data movement" instructions):
  32x32b.xN    a warp reads 32 TMEM lanes (its own sub-partition), N consecutive
               32-bit columns per lane; thread i gets lane i.
  16x32bx2.xN  a warp reads 16 lanes twice: threads 0-15 get lanes 0-15 of the
               sub-partition at columns [col, col+N), threads 16-31 the same lanes at
               columns [col+half, col+half+N); `half` is an immediate. This is the
               natural read of an M=64 accumulator, whose rows sit in lanes 0-15 of
               each sub-partition.

Run:  python split_kv_sparse_gb300/csrc/gen_tmem_ldst.py
"""
from pathlib import Path


def _regs(n, start=0):
    return ", ".join(f"%{i}" for i in range(start, start + n))


def _outs(n, mode):
    items = [f'"{mode}"(r[{i}])' for i in range(n)]
    return ",\n      ".join(", ".join(items[i:i + 8]) for i in range(0, n, 8))


def ld_32x32b(n):
    return f"""__device__ __forceinline__ void tmem_ld_32x32b_x{n}(uint32_t taddr, uint32_t (&r)[{n}]) {{
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x{n}.b32 {{{_regs(n)}}}, [%{n}];"
      : {_outs(n, "=r")}
      : "r"(taddr));
}}
"""


def ld_16x32bx2(n, half):
    return f"""__device__ __forceinline__ void tmem_ld_16x32bx2_x{n}_h{half}(uint32_t taddr, uint32_t (&r)[{n}]) {{
  asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x{n}.b32 {{{_regs(n)}}}, [%{n}], {half};"
      : {_outs(n, "=r")}
      : "r"(taddr));
}}
"""


def st_32x32b(n):
    return f"""__device__ __forceinline__ void tmem_st_32x32b_x{n}(uint32_t taddr, const uint32_t (&r)[{n}]) {{
  asm volatile("tcgen05.st.sync.aligned.32x32b.x{n}.b32 [%0], {{{_regs(n, 1)}}};"
      :: "r"(taddr),
      {_outs(n, "r")}
      : "memory");
}}
"""


def wait_ld(n):
    return f"""// Waits for this thread's TMEM loads; threading the registers through the asm keeps
// every use of them after the wait.
__device__ __forceinline__ void tmem_wait_ld_x{n}(uint32_t (&r)[{n}]) {{
  asm volatile("tcgen05.wait::ld.sync.aligned;"
      : {_outs(n, "+r")}
      :: "memory");
}}
"""


def main():
    parts = ["// Inline-PTX wrappers for tcgen05.ld / tcgen05.st (written by gen_tmem_ldst.py).\n"]
    parts += [ld_32x32b(16), ld_32x32b(32), ld_32x32b(64), ld_16x32bx2(32, 32), ld_16x32bx2(16, 32),
              ld_16x32bx2(64, 64)]
    parts += [wait_ld(16), wait_ld(32), wait_ld(64)]
    parts += [st_32x32b(16), st_32x32b(32), st_32x32b(64)]
    out = Path(__file__).with_name("tmem_ldst.inc")
    out.write_text("\n".join(parts))


if __name__ == "__main__":
    main()
