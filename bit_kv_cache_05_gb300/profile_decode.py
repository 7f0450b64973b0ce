"""Profiling driver: build one cache of a named workload and run a few
decode launches (for ncu captures of the decode kernel).

  python bit_kv_cache_05_gb300/profile_decode.py pages_S65536 3
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv):
    import torch
    from bit_kv_cache_05_gb300 import synth
    from bit_kv_cache_05_gb300.cache import KiviCache
    name = argv[1] if len(argv) > 1 else "pages_S65536"
    n = int(argv[2]) if len(argv) > 2 else 3
    w = synth.workload(name)
    inp = synth.make_inputs(w, device="cuda")
    c = KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=w.bits,
                  group=w.group, residual=w.residual, max_seq=w.max_seq)
    del inp["K"], inp["V"]
    torch.cuda.synchronize()
    for _ in range(n):
        out = c.decode_attend(inp["q"])
    torch.cuda.synchronize()
    c.device_status()
    print("ok", name, c.decode_kernel(), float(out.abs().max()))
    c.close()


if __name__ == "__main__":
    main(sys.argv)
