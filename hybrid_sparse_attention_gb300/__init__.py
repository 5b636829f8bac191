"""GB300-native decode-time hybrid sparse attention (SWA + C4/C128)."""
