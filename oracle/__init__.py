"""CPU oracle for one DFlash draft-and-verify step — TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` may
import or run anything in this package. The library's product path never does,
and shares no code with it: this package imports neither the CUDA extension nor
its binding, and the CUDA side imports nothing from here.

Sources (web pages describing DFlash; cited by site and section):
  jansverre.net   "DFlash: slik kan spekulativ dekoding gi opptil 6x raskere AI-inferens"
  bpdata.com      Hungarian news article on DFlash block-diffusion speculative decoding
  theaistack.guide "DFlash Crea Blocchi Interi di Token Contemporaneamente, Aumentando Fino
                   a 15x la Velocità su NVIDIA Blackwell"
  7minutos.es     "La decodificación especulativa de DFlash elabora bloques de tokens
                   completos en paralelo ..."

Modules:
  dflash_ref  the step, written out in the pages' order with NumPy (fp64 by default)
  naive       an independent per-slot scalar-loop recomputation for tiny shapes, used
              as a brute-force pin of dflash_ref

Pinning status: verify is pinned exactly (brute force over agreement masks, closed
cases). RMSNorm, RoPE, attention and SwiGLU are pinned by closed forms and by
library routines called from the tests. The draft forward as a whole is pinned
against `naive` and the injection against its own associativity. The pages print
no intermediate values, so the architectural readings (norm placement, RoPE
convention, eps) are pinned only as readings, not by the pages.
"""
