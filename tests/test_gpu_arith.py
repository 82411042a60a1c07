"""The quantizer's fast arithmetic against the IEEE operations it replaces,
checked exhaustively on the GPU through the library's testing hook:

  * the scale (max - min) / (2^b - 1) by Markstein's corrected product by the
    reciprocal must equal the IEEE divide for every float of the quantizer's
    domain: 0 and the differences of fp16 values (2^-24 .. 131008);
  * the hardware reciprocal of the scale must stay within 2 ulp (2^-22
    relative) over every positive finite fp16 value: the codes' near-tie window
    (1e-5 around half-integers, quotients at most 15.008) is sized for a
    product dx * rcp(s) within 3 ulp of the IEEE quotient.
The bit-exact packing tests then hold the whole quantizer to the oracle."""

import pytest

from bit_quantized_kv_pack_gb300 import kvq

pytestmark = pytest.mark.gpu


def test_constant_division_and_reciprocal_are_exact_enough():
    div, rcp_worst = kvq.kvq_testing_check_arithmetic()
    for k, (all_floats, domain) in zip((15, 7, 3), div):
        print(f"divisor {k}: {all_floats} mismatches over all non-negative floats, "
              f"{domain} in the quantizer's domain")
        assert domain == 0, (k, all_floats, domain)
    assert rcp_worst <= 2.0 ** -22, rcp_worst
