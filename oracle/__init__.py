"""CPU oracle for the V-JEPA 2 / 2.1 video ViT encoder forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
run this package: only the tests, the smoke check and the benchmark's CPU
baseline leg do.  It shares no code with the CUDA library.

Every function restates one step of the method as the pages define it, in
float64, with library primitives (matmul, erf, exp) as the only building
blocks and no blocking, fusion or reordering beyond the definition.
"""
from .encoder import (  # noqa: F401
    IMAGENET_MEAN, IMAGENET_STD,
    normalise_clip, patch_embed, token_positions, rope_split, rope_tables,
    rot90_pairs, apply_rope, layer_norm, gelu_erf, attention_heads,
    block_forward, block_forward_rows, encoder_forward, predictor_forward,
    grid_positions_from_ids, predictor_input, encoder_rope, encoder_embed, is_image,
    predictor_outputs, attentive_pool_forward,
)
