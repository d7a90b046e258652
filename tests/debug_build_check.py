"""Runs the debug build of libmla_decode (bounds-checked kernels) on a set of
shapes covering every kernel variant and reports, as one JSON line, the error
word and the parity of each call.  Invoked in a fresh process by
tests/test_gpu_debug_build.py (the debug library is the only one it loads)."""
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from mla_decode_attention_08_gb300 import binding  # noqa: E402
from mla_decode_attention_08_gb300.build import build  # noqa: E402
from mla_decode_attention_08_gb300.inputs import make_from_lengths  # noqa: E402
from oracle.attention import bf16_bits_to_f64, mla_decode_ref_bf16kv  # noqa: E402
from tests.gpu_util import DeviceCase, OracleCase, bits_to_bf16, compare  # noqa: E402
from tests.test_gpu_mxfp4 import MxCase  # noqa: E402


def main() -> None:
    binding.load_library(build(debug=True))
    results = {}
    lengths = [1, 127, 128, 129, 700, 0, 3000, 5]
    for paged in (False, True):
        for qo_len in (1, 2, 4):
            inp = make_from_lengths(lengths, seed=70 + qo_len, paged=paged, qo_len=qo_len)
            dev = DeviceCase(inp)
            for sms in (3, 152):
                gpu, err, _, _ = dev.run(sms=sms)
                st = compare(gpu, OracleCase(inp).reference())
                results[f"e4m3 paged={paged} q={qo_len} sms={sms}"] = {"err": err, **st}
    inp = make_from_lengths(lengths, seed=80, qo_len=2)
    q = bits_to_bf16(inp.q_bits)
    kv = bits_to_bf16(inp.kv_bits)
    qo, kvp = torch.from_numpy(inp.qo_indptr).cuda(), torch.from_numpy(inp.kv_indptr).cuda()
    out = torch.empty((inp.batch * 2, 16, 512), dtype=torch.bfloat16, device="cuda")
    plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, 5, qo_len=2)
    ws = binding.new_workspace(plan)
    binding.mla_decode_fwd_bf16kv(q, kv, qo, kvp, out, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    ref = mla_decode_ref_bf16kv(bf16_bits_to_f64(inp.q_bits), inp.kv_bits, inp.qo_indptr, inp.kv_indptr)
    results["bf16 q=2"] = {"err": binding.mla_decode_read_error(ws), **compare(out.float().cpu().numpy(), ref)}
    # the cluster split (e4m3 and bf16 caches, sizes 8, 4 and 2)
    for size_lengths, sms in (([1024, 1, 0, 700], 152), (list(range(3, 1024, 37)), 152),
                              ([300, 299, 1], 152)):
        inp = make_from_lengths(size_lengths, seed=82, max_kv_len=max(size_lengths))
        dev = DeviceCase(inp)
        gpu, err, plan, _ = dev.run(sms=sms)
        st = compare(gpu, OracleCase(inp).reference())
        results[f"e4m3 cluster={plan.cluster}"] = {"err": err, **st}
        q, kv = bits_to_bf16(inp.q_bits), bits_to_bf16(inp.kv_bits)
        qo, kvp = torch.from_numpy(inp.qo_indptr).cuda(), torch.from_numpy(inp.kv_indptr).cuda()
        out = torch.empty((inp.batch, 16, 512), dtype=torch.bfloat16, device="cuda")
        ws = binding.new_workspace(plan)
        binding.mla_decode_fwd_bf16kv(q, kv, qo, kvp, out, plan=plan, workspace=ws)
        torch.cuda.synchronize()
        ref = mla_decode_ref_bf16kv(bf16_bits_to_f64(inp.q_bits), inp.kv_bits, inp.qo_indptr,
                                    inp.kv_indptr)
        results[f"bf16 cluster={plan.cluster}"] = {"err": binding.mla_decode_read_error(ws),
                                                   **compare(out.float().cpu().numpy(), ref)}
    inp = make_from_lengths(lengths, seed=81)
    case = MxCase(inp)
    for sms in (3, 152):
        gpu, err, _, _ = case.run(sms=sms)
        results[f"mxfp4 sms={sms}"] = {"err": err, **compare(gpu, case.reference())}
    print(json.dumps(results))


if __name__ == "__main__":
    main()
