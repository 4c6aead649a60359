"""CPU oracle pinned to facts outside itself (see oracle_pins.py for each pin's source)."""
import oracle_pins as P


def test_statistics_closed_form():
    P.pin_statistics_closed_form()


def test_klt_known_spectrum():
    P.pin_klt_known_spectrum()


def test_transform_preserves_inner_products():
    P.pin_transform_preserves_inner_products()


def test_sixteen_bits_preserve_attention():
    P.pin_sixteen_bits_preserve_attention()


def test_key_distortion_monte_carlo():
    P.pin_key_distortion_monte_carlo()


def test_value_distortion_monte_carlo():
    P.pin_value_distortion_monte_carlo()


def test_additive_key_value_distortion():
    P.pin_additive_key_value_distortion()


def test_water_fill_golden():
    P.pin_water_fill_golden()


def test_water_fill_kkt():
    P.pin_water_fill_kkt()


def test_water_fill_integer_properties():
    P.pin_water_fill_integer_properties()


def test_water_fill_vs_brute_force():
    worst = P.pin_water_fill_vs_brute_force()
    print(f"worst integer-rounding distortion ratio vs exhaustive optimum: {worst:.4f}")


def test_compression_accounting():
    P.pin_compression_accounting()


def test_quantize_pack_golden():
    P.pin_quantize_pack_golden()


def test_pack_roundtrip():
    P.pin_pack_roundtrip()


def test_layout_fit_golden():
    P.pin_layout_fit_golden()


def test_token_pack_golden():
    P.pin_token_pack_golden()


def test_token_layout_fit_golden():
    P.pin_token_layout_fit_golden()


def test_layout_fit_properties():
    worst = P.pin_layout_fit_properties()
    print(f"worst distortion ratio of the fitted layout vs the unconstrained allocation: {worst:.4f}")


def test_quantizer_error_bound():
    P.pin_quantizer_error_bound()


def test_zero_bit_channels_are_the_mean():
    P.pin_zero_bit_channels_are_the_mean()


def test_half_conversion():
    P.pin_half_conversion()


def test_decode_brute_force():
    P.pin_decode_brute_force()


def test_calibrate_structure():
    P.pin_calibrate_structure()


def test_storage_order():
    P.pin_storage_order()


def test_exchange_rate_monte_carlo():
    P.pin_exchange_rate_monte_carlo()


def test_joint_split_by_enumeration():
    P.pin_joint_split_by_enumeration()


def test_aware_basis_commuting():
    P.pin_aware_basis_commuting()


def test_aware_basis_two_channels():
    P.pin_aware_basis_two_channels()


def test_aware_basis_bounds():
    P.pin_aware_basis_bounds()


def test_whitened_key_transform():
    P.pin_whitened_key_transform()


def test_rotary_embedding():
    P.pin_rotary_embedding()


def test_token_weights():
    P.pin_token_weights()


def test_token_keep():
    P.pin_token_keep()


def test_compact():
    P.pin_compact()
