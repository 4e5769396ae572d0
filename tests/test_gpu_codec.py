"""Codec quantizer decode (lookup-and-sum) through the C ABI vs the oracle: bit-exact, since both
add the same bf16 rows in codebook order in fp32."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ncb,cbs,dim,n", [(10, 4096, 1024, 256), (1, 64, 264, 1), (7, 300, 8, 33)])
def test_codec_latent_bit_exact(ncb, cbs, dim, n):
    import dual_ar_tts_gb300 as pkg
    qs = synth.codec_quantizers(5, ncb, cbs, dim)
    codes = synth.uniform_int(6, 7, ncb * n, 0, cbs - 1)
    dq = [torch.from_numpy(q.view(np.int16)).cuda() for q in qs]
    dc = torch.from_numpy(codes).cuda()
    lat = torch.full((n, dim), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkg.s2_codec_latent(ncb, cbs, dim, [t.data_ptr() for t in dq], n, dc.data_ptr(), lat.data_ptr(), st.data_ptr())
    torch.cuda.synchronize()
    assert int(st[0]) == pkg.S2_OK
    np.testing.assert_array_equal(lat.cpu().numpy(), oracle.codec_latent(qs, codes, n))


def test_codec_latent_flags_out_of_range_codes():
    import dual_ar_tts_gb300 as pkg
    ncb, cbs, dim, n = 3, 64, 16, 4
    qs = synth.codec_quantizers(5, ncb, cbs, dim)
    codes = synth.uniform_int(6, 7, ncb * n, 0, cbs - 1)
    codes[1 * n + 2] = cbs  # codebook 1, frame 2
    dq = [torch.from_numpy(q.view(np.int16)).cuda() for q in qs]
    lat = torch.zeros((n, dim), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkg.s2_codec_latent(ncb, cbs, dim, [t.data_ptr() for t in dq], n, torch.from_numpy(codes).cuda().data_ptr(),
                        lat.data_ptr(), st.data_ptr())
    torch.cuda.synchronize()
    assert int(st[0]) == pkg.S2_EINVAL
    ok = codes.copy()
    ok[1 * n + 2] = 0
    want = oracle.codec_latent(qs, ok, n)
    got = lat.cpu().numpy()
    np.testing.assert_array_equal(np.delete(got, 2, axis=0), np.delete(want, 2, axis=0))
